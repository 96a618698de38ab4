// k_gemm.cu - the encoder's two tensor-core GEMMs (ResidualKV notes §2.3, §2.4).
//
//   GEMM-1/2:  [kv; mean] rows x [W_c1 | W_c2]  ->  h = Swish(a1) * a2, then the
//              difference h(kv) - h(mean) of each token in fp32, stored as two bf16 parts
//              D = [d_hi | d_lo] (d_hi = RN_bf16(d), d_lo = RN_bf16(d - d_hi): together
//              d to about 2^-18 relative).
//              A tile m (128 rows) = the bf16 kv rows of dense rows q = 64 m .. 64 m + 63
//              (the first 2d_k columns of the query rows Q, or their dense copy Qd when a
//              pass holds several sequences) over their bf16 mean rows (M), two 64-row
//              TMA boxes into one swizzled stage;
//              B = W12 [2 d_ff, 2d_k] with gate and value columns interleaved per
//              256-row tile so that one 128x256 accumulator holds a1 and a2 of the same
//              128 hidden units.  The epilogue threads of a token's kv row and mean row
//              swap their fp32 h through shared memory and each forms half of the row's d.
//   GEMM-3:    D viewed as [m, 2 d_ff] (row q = [d_hi | d_lo]) x [W_c3; W_c3]
//              -> z_q = d_q W_c3 = h(kv_q) W_c3 - h(mean_q) W_c3.  Each f_c keeps its own
//              nonlinear map (never f_c of a difference, ResidualKV notes §2.3 boxed z);
//              W_c3 is linear, so subtracting the mapped rows before or after it is the
//              same value, and subtracting them first in fp32 keeps the bf16 rounding of
//              the tensor-core operand off each f_c output.
//              The epilogue quantises each 32-column group in the thread that owns the
//              token row (min/max, FP16 extremes rounded outward, Delta, round-half-
//              even, clamp, nibble/crumb packing) and writes codes and extremes.
//
// Both run one persistent CTA per SM: a 4..6-stage TMA ring feeds tcgen05.mma (M=128,
// K=16 per instruction, fp32 accumulators in TMEM), two TMEM accumulators let the
// epilogue of tile t overlap the main loop of tile t+1.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc_common.cuh"

namespace rkv {
namespace {

struct GemmShape {
  int m_tiles, n_tiles, nkb;  // tiles of 128 rows, tiles of BN columns, 64-wide k-blocks
  int b_kwrap;                // B's k-block coordinate is kb % b_kwrap
  int* status;
  const int32_t* m_list;      // if set, row tile i is m_list[i] (device), else i
};

__device__ __forceinline__ int row_tile(const GemmShape& g, int i) {
  return g.m_list ? g.m_list[i] : i;
}

struct Epi12Args {
  __nv_bfloat16* H;
  int dff;
  int rows;  // dense rows (kv and mean row pairs)
};

// mean_precompute, reference pre-activations: P[row] = r [W_c1 | W_c2] in fp32
struct EpiPArgs {
  float* P;
  int64_t rows;  // B R_cap pool rows
  int ld;        // 2 d_ff
};

// mean_precompute, GEMM-1/2 over kv rows only
struct Epi12RArgs {
  __nv_bfloat16* H;
  int dff;
  int rows;                // dense rows
  const int32_t* q_dst;    // per dense row: storage row (seq T_cap + pos)
  const int32_t* ref_idx;  // [B T_cap, topk] pool slots of each token
  int topk, R_cap, T_cap;
  const float* P;
  int zero_row;            // a row of P that holds zeros (stands in for a missing slot)
};

struct Epi3Args {
  const int32_t* q_dst;  // per dense row: storage row
  int rows;              // dense rows
  uint8_t* codes;
  uint32_t* meta;
  int code_bytes, G, bits, BN;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat16 lo = __float2bfloat16_rn(a), hi = __float2bfloat16_rn(b);
  return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}

// ---------------------------------------------------------------- epilogues
struct Epi12 {
  using Args = Epi12Args;
  static constexpr bool kSplitA = true;
  static constexpr uint32_t kExchangeBytes = kTileM * 32 * 4;   // 128 rows x 32 fp32
  // Tile row i holds the kv (i < 64) or mean (i >= 64) row of dense row 64 m + i % 64.
  // Per 32-column chunk: every thread writes its row's fp32 h to the exchange buffer,
  // then the kv thread of token t forms d = h(kv) - h(mean) for the chunk's first 16
  // columns and the mean thread of t for the last 16, and stores d_hi and d_lo.
  __device__ static void run(const Args& a, uint32_t tacc, int m, int n, int row_in_tile,
                             int* status, float* xch) {
    const int half = row_in_tile >= kTileM / 2 ? 1 : 0;
    const int tok = row_in_tile & (kTileM / 2 - 1);
    const int64_t q = (int64_t)m * (kTileM / 2) + tok;
    const bool valid = q < a.rows;
    // exchange rows of 32 floats; the 16-byte chunks of row r sit at chunk ^ (r & 7) so
    // that a warp's 16-byte accesses to 32 consecutive rows spread over the banks
    float4* my_row = reinterpret_cast<float4*>(xch) + row_in_tile * 8;
    const float4* kv_row = reinterpret_cast<const float4*>(xch) + tok * 8;
    const float4* mn_row = reinterpret_cast<const float4*>(xch) + (tok + kTileM / 2) * 8;
    const int sw_me = row_in_tile & 7, sw_tok = tok & 7;   // (tok + 64) & 7 == tok & 7
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t g[32], v[32];
      tmem_ld32(tacc + c * 32, g);
      tmem_ld32(tacc + 128 + c * 32, v);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float a1 = __uint_as_float(g[4 * i + j]);
          const float a2 = __uint_as_float(v[4 * i + j]);
          h[j] = __fdividef(a1, 1.0f + __expf(-a1)) * a2;   // Swish (beta = 1) times a2
        }
        my_row[i ^ sw_me] = make_float4(h[0], h[1], h[2], h[3]);
      }
      bar_sync(1, 128);
      uint32_t whi[8], wlo[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int ch = 4 * half + i;                  // this thread's 16-byte chunks
        const float4 hk = kv_row[ch ^ sw_tok], hm = mn_row[ch ^ sw_tok];
        const float d[4] = {hk.x - hm.x, hk.y - hm.y, hk.z - hm.z, hk.w - hm.w};
        float lo[4];
        uint32_t hb[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          hb[j] = pack_bf16x2(d[2 * j], d[2 * j + 1]);
          lo[2 * j] = d[2 * j] - __uint_as_float(hb[j] << 16);
          lo[2 * j + 1] = d[2 * j + 1] - __uint_as_float(hb[j] & 0xFFFF0000u);
        }
        whi[2 * i] = hb[0];
        whi[2 * i + 1] = hb[1];
        wlo[2 * i] = pack_bf16x2(lo[0], lo[1]);
        wlo[2 * i + 1] = pack_bf16x2(lo[2], lo[3]);
      }
      if (valid) {
        __nv_bfloat16* dst = a.H + q * (2 * (int64_t)a.dff) + (int64_t)n * 128 + c * 32 + half * 16;
        uint4* dh = reinterpret_cast<uint4*>(dst);
        uint4* dl = reinterpret_cast<uint4*>(dst + a.dff);
        dh[0] = make_uint4(whi[0], whi[1], whi[2], whi[3]);
        dh[1] = make_uint4(whi[4], whi[5], whi[6], whi[7]);
        dl[0] = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
        dl[1] = make_uint4(wlo[4], wlo[5], wlo[6], wlo[7]);
      }
      bar_sync(1, 128);                                // the buffer is reused next chunk
    }
  }
};

// The fp32 accumulators of 128 pool rows x 256 columns (one W12 tile: 128 W_c1 then 128
// W_c2 columns) stored as they are: row r of tile m is pool row 128 m + r.
struct EpiP {
  using Args = EpiPArgs;
  static constexpr bool kSplitA = false;
  static constexpr uint32_t kExchangeBytes = 0;
  __device__ static void run(const Args& a, uint32_t tacc, int m, int n, int row_in_tile,
                             int*, float*) {
    const int64_t row = (int64_t)m * kTileM + row_in_tile;
    const bool valid = row < a.rows;
    float* dst = a.P + row * a.ld + (int64_t)n * 256;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      uint32_t r[32];
      tmem_ld32(tacc + c * 32, r);
      tmem_ld_wait();
      if (!valid) continue;
      float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        d4[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                            __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
    }
  }
};

// GEMM-1/2 of 128 kv rows with the mean's hidden row taken from the references'
// pre-activations: per token, the k_i pool slots' P rows summed over the tile's 128 hidden
// units (gate and value columns), scaled by 1 / k_i (exact for k_i = 1, 2, 4; a correctly
// rounded division for 3), and put through the same SwiGLU as the kv row; the thread of
// token row q stores d = h(kv) - h(mean) as [d_hi | d_lo].
// The gathers are cooperative: per 32-column chunk, a warp reads the P slices of its 32
// tokens as whole 128-byte rows (lane l: token 4 i + l / 8, columns 4 (l % 8) ..), four
// tokens per 16-byte load instruction, forms h(mean) column-wise into shared memory
// (rows padded to 36 floats), and each thread then reads its own row back.
struct Epi12R {
  using Args = Epi12RArgs;
  static constexpr bool kSplitA = false;
  static constexpr int kRowF = 36;                           // padded h(mean) row, floats
  static constexpr uint32_t kWarpBytes = 32 * kRowF * 4 + 32 * 4 * 4 + 32 * 4;
  static constexpr uint32_t kExchangeBytes = 4 * kWarpBytes;
  __device__ static void run(const Args& a, uint32_t tacc, int m, int n, int row_in_tile,
                             int*, float* xch) {
    const int ew = row_in_tile >> 5, l = row_in_tile & 31;
    float* hm_s = xch + ew * (kWarpBytes / 4);               // [32][kRowF]
    int* prow_s = reinterpret_cast<int*>(hm_s + 32 * kRowF);  // [32][4] P rows (zero row if none)
    float* kinv_s = reinterpret_cast<float*>(prow_s + 32 * 4);  // [32]: 1/k, or -3 for k = 3
    const int64_t q = (int64_t)m * kTileM + row_in_tile;
    const bool valid = q < a.rows;
    {
      int pr[4] = {a.zero_row, a.zero_row, a.zero_row, a.zero_row};
      int k = 0;
      if (valid) {
        const int64_t dst = a.q_dst[q];
        const int base = (int)(dst / a.T_cap) * a.R_cap;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int slot = t < a.topk ? a.ref_idx[dst * a.topk + t] : -1;
          if (slot >= 0 && slot < a.R_cap) pr[k++] = base + slot;
        }
      }
      reinterpret_cast<int4*>(prow_s)[l] = make_int4(pr[0], pr[1], pr[2], pr[3]);
      kinv_s[l] = k == 3 ? -3.0f : (k == 2 ? 0.5f : (k == 4 ? 0.25f : 1.0f));
    }
    __syncwarp();
    const int sub = l >> 3, c4 = (l & 7) * 4;                // token within a group of 4, column
    const int64_t ld = 2 * (int64_t)a.dff;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t g[32], v[32];
      tmem_ld32(tacc + c * 32, g);
      tmem_ld32(tacc + 128 + c * 32, v);
      // h(mean) of the warp's 32 tokens, columns c4 .. c4 + 3 of this chunk
      const int64_t col = (int64_t)n * 256 + c * 32 + c4;
#pragma unroll 4
      for (int i = 0; i < 8; ++i) {
        const int j = 4 * i + sub;
        const int4 pr = reinterpret_cast<const int4*>(prow_s)[j];
        const int prs[4] = {pr.x, pr.y, pr.z, pr.w};
        float4 sg = make_float4(0.f, 0.f, 0.f, 0.f), sv = sg;
#pragma unroll
        for (int t = 0; t < 4; ++t) {              // missing slots read the zero row
          const float* base = a.P + (int64_t)prs[t] * ld + col;
          const float4 x = __ldg(reinterpret_cast<const float4*>(base));
          const float4 y = __ldg(reinterpret_cast<const float4*>(base + 128));
          sg.x += x.x, sg.y += x.y, sg.z += x.z, sg.w += x.w;
          sv.x += y.x, sv.y += y.y, sv.z += y.z, sv.w += y.w;
        }
        const float kv = kinv_s[j];
        const float s1[4] = {sg.x, sg.y, sg.z, sg.w}, s2[4] = {sv.x, sv.y, sv.z, sv.w};
        float h[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float m1 = kv < 0.f ? __fdiv_rn(s1[e], 3.0f) : s1[e] * kv;
          const float m2 = kv < 0.f ? __fdiv_rn(s2[e], 3.0f) : s2[e] * kv;
          h[e] = __fdividef(m1, 1.0f + __expf(-m1)) * m2;
        }
        *reinterpret_cast<float4*>(hm_s + j * kRowF + c4) = make_float4(h[0], h[1], h[2], h[3]);
      }
      __syncwarp();
      tmem_ld_wait();
      uint32_t whi[16], wlo[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 hm = *reinterpret_cast<const float4*>(hm_s + l * kRowF + 4 * i);
        const float hms[4] = {hm.x, hm.y, hm.z, hm.w};
        float d[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a1 = __uint_as_float(g[4 * i + e]), a2 = __uint_as_float(v[4 * i + e]);
          d[e] = __fdividef(a1, 1.0f + __expf(-a1)) * a2 - hms[e];
        }
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const uint32_t hb = pack_bf16x2(d[e], d[e + 1]);
          whi[2 * i + e / 2] = hb;
          wlo[2 * i + e / 2] = pack_bf16x2(d[e] - __uint_as_float(hb << 16),
                                           d[e + 1] - __uint_as_float(hb & 0xFFFF0000u));
        }
      }
      __syncwarp();                                    // hm_s is rewritten next chunk
      if (!valid) continue;
      __nv_bfloat16* dst = a.H + q * (2 * (int64_t)a.dff) + (int64_t)n * 128 + c * 32;
      uint4* dh = reinterpret_cast<uint4*>(dst);
      uint4* dl = reinterpret_cast<uint4*>(dst + a.dff);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        dh[i] = make_uint4(whi[4 * i], whi[4 * i + 1], whi[4 * i + 2], whi[4 * i + 3]);
        dl[i] = make_uint4(wlo[4 * i], wlo[4 * i + 1], wlo[4 * i + 2], wlo[4 * i + 3]);
      }
    }
  }
};

// Quantise one 32-value group held by this thread and write its code bytes and extremes.
__device__ __forceinline__ void quant_group(const float* z, int bits, uint8_t* code, uint32_t* meta,
                                            int* status) {
  if (bits == 16) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(z[2 * i], z[2 * i + 1]);
    uint4* d = reinterpret_cast<uint4*>(code);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    *meta = 0u;
    return;
  }
  float zmin = z[0], zmax = z[0];
#pragma unroll
  for (int i = 1; i < 32; ++i) {
    zmin = fminf(zmin, z[i]);
    zmax = fmaxf(zmax, z[i]);
  }
  const bool sat = (fabsf(zmin) > 65504.0f) || (fabsf(zmax) > 65504.0f);
  if (sat) atomicOr(status, RKV_FLAG_FP16_SAT);
  __half lo16, hi16;
  const bool constant = (zmin == zmax);
  if (constant) {
    lo16 = __float2half_rn(fminf(fmaxf(zmin, -65504.0f), 65504.0f));
    hi16 = lo16;
  } else {
    lo16 = __float2half_rd(fmaxf(zmin, -65504.0f));
    hi16 = __float2half_ru(fminf(zmax, 65504.0f));
  }
  const float lo = __half2float(lo16), hi = __half2float(hi16);
  const int levels = (1 << bits) - 1;
  const float delta = __fdiv_rn(__fsub_rn(hi, lo), (float)levels);
  const bool zero = constant || (delta == 0.0f);
  // (z - min) / Delta as a product with the correctly rounded reciprocal: the pre-round
  // value moves by at most ~2 ulp, which can change a code only within ~1e-6 of a .5
  // boundary (the method's code tolerance allows +-1 within 1e-3 of one)
  const float rdelta = zero ? 0.0f : __frcp_rn(delta);
  int q[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    int v = zero ? 0 : __float2int_rn(__fmul_rn(__fsub_rn(z[i], lo), rdelta));
    q[i] = v < 0 ? 0 : (v > levels ? levels : v);
  }
  if (bits == 4) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t x = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) x |= (uint32_t)q[8 * k + i] << (4 * i);
      w[k] = x;
    }
    *reinterpret_cast<uint4*>(code) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {  // bits == 2
    uint32_t w[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      uint32_t x = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) x |= (uint32_t)q[16 * k + i] << (2 * i);
      w[k] = x;
    }
    *reinterpret_cast<uint2*>(code) = make_uint2(w[0], w[1]);
  }
  *meta = (uint32_t)__half_as_ushort(lo16) | ((uint32_t)__half_as_ushort(hi16) << 16);
}

struct Epi3 {
  using Args = Epi3Args;
  static constexpr bool kSplitA = false;
  static constexpr uint32_t kExchangeBytes = 0;
  __device__ static void run(const Args& a, uint32_t tacc, int m, int n, int row_in_tile,
                             int* status, float*) {
    const int64_t row = (int64_t)m * kTileM + row_in_tile;
    const int64_t dst = row < a.rows ? (int64_t)a.q_dst[row] : -1;
    const bool valid = dst >= 0;                     // padding rows are not stored
    const int groups = a.BN / 32;
#pragma unroll 1
    for (int gi = 0; gi < groups; ++gi) {
      uint32_t r[32];
      tmem_ld32(tacc + gi * 32, r);
      tmem_ld_wait();
      if (!valid) continue;
      float z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = __uint_as_float(r[i]);
      const int g = n * groups + gi;   // group index within the token
      uint8_t* code = a.codes + dst * a.code_bytes + (int64_t)g * (a.bits * 32 / 8);
      uint32_t* meta = a.meta + dst * a.G + g;
      quant_group(z, a.bits, code, meta, status);
    }
  }
};

// ---------------------------------------------------------------- kernel
template <int BN, int STAGES, typename Epi>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                   const __grid_constant__ CUtensorMap tmB, GemmShape g, typename Epi::Args ea) {
  constexpr uint32_t kBBytes = BN * 128;
  constexpr uint32_t kTmemCols = 2 * BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * kTileABytes;
  float* xch = reinterpret_cast<float*>(sB + STAGES * kBBytes);   // epilogue exchange
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * kBBytes + Epi::kExchangeBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int n_tiles_total = g.m_tiles * g.n_tiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);                        // one arrival per epilogue warp
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch(&tmA);
    if (Epi::kSplitA) tma_prefetch(&tmA2);
    tma_prefetch(&tmB);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (elect_one()) {
      Ring ring;
      int issued[STAGES];
      uint32_t issued_phase[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = 0, issued_phase[s] = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < n_tiles_total && ok; t += gridDim.x) {
        const int m = row_tile(g, t / g.n_tiles), n = t % g.n_tiles;
        for (int kb = 0; kb < g.nkb; ++kb) {
          if (!mbar_wait(&empty[ring.stage], ring.phase ^ 1u, abort_flag, g.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[ring.stage], kTileABytes + kBBytes);
          if (Epi::kSplitA) {
            // rows 0..63 from tmA, rows 64..127 from tmA2 (the same 64 retrieval rows)
            tma_load_2d(sA + ring.stage * kTileABytes, &tmA, &full[ring.stage], kb * kTileK,
                        m * (kTileM / 2));
            tma_load_2d(sA + ring.stage * kTileABytes + kTileABytes / 2, &tmA2, &full[ring.stage],
                        kb * kTileK, m * (kTileM / 2));
          } else {
            tma_load_2d(sA + ring.stage * kTileABytes, &tmA, &full[ring.stage], kb * kTileK,
                        m * kTileM);
          }
          const int kbB = kb % g.b_kwrap;
          for (int h = 0; h < BN; h += 256)
            tma_load_2d(sB + ring.stage * kBBytes + h * 128, &tmB, &full[ring.stage],
                        kbB * kTileK, n * BN + h);
          issued[ring.stage] = 1;
          issued_phase[ring.stage] = ring.phase;
          ring.next(STAGES);
        }
      }
      if (!ok) {
        for (int s = 0; s < STAGES; ++s)
          if (issued[s]) drain_wait(&full[s], issued_phase[s]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t idesc = idesc_bf16_f32(kTileM, BN > 256 ? 256 : BN);
      Ring ring;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool any = false;
      int last_stage = 0;
      uint32_t last_phase = 0;
      for (int t = blockIdx.x; t < n_tiles_total && ok; t += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, g.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        for (int kb = 0; kb < g.nkb; ++kb) {
          if (!mbar_wait(&full[ring.stage], ring.phase, abort_flag, g.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + ring.stage * kTileABytes);
          const uint32_t b0 = smem_u32(sB + ring.stage * kBBytes);
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k) {
            for (int h = 0; h < BN; h += 256)
              umma_bf16(d + h, sdesc_sw128(a0 + k * 32), sdesc_sw128(b0 + h * 128 + k * 32),
                        idesc, (kb | k) != 0 ? 1u : 0u);
          }
          umma_commit(&empty[ring.stage]);
          any = true;
          last_stage = ring.stage;
          last_phase = ring.phase;
          ring.next(STAGES);
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok && any) drain_wait(&empty[last_stage], last_phase);
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------ epilogue
    const int ew = warp - kEpiWarp0;
    const int row_in_tile = ew * 32 + (int)lane_id();
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < n_tiles_total; t += gridDim.x) {
      const int m = row_tile(g, t / g.n_tiles), n = t % g.n_tiles;
      // An epilogue that swaps rows between its warps (named barriers inside) goes on
      // only if all four warps' waits succeeded, so no warp is left alone at a barrier.
      bool ok = warp_wait(&tfull[acc], acc_phase, abort_flag, g.status);
      if (Epi::kExchangeBytes > 0) ok = bar_red_and(2, 128, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tacc = tmem + ((uint32_t)(ew * 32) << 16) + (uint32_t)(acc * BN);
      Epi::run(ea, tacc, m, n, row_in_tile, g.status, xch);
      tc_fence_before();
      __syncwarp();
      if (lane_id() == 0) mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int BN, int STAGES, typename Epi>
constexpr size_t gemm_smem_bytes() {
  return 1024 + (size_t)STAGES * (kTileABytes + BN * 128) + Epi::kExchangeBytes +
         8 * (2 * STAGES + 4) + 16;
}

template <int BN, int STAGES, typename Epi>
cudaError_t run_gemm(rkv_ctx* c, const CUtensorMap& tA, const CUtensorMap& tA2, const CUtensorMap& tB,
                     GemmShape g, typename Epi::Args ea, const char* name, cudaStream_t s) {
  const size_t smem = gemm_smem_bytes<BN, STAGES, Epi>();
  auto kern = tc_gemm_kernel<BN, STAGES, Epi>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int tiles = g.m_tiles * g.n_tiles;
  if (tiles == 0) return cudaSuccess;
  const int grid = tiles < c->num_sms ? tiles : c->num_sms;
  cudaEvent_t ev;
  timing_begin(c, name, s, &ev);
  kern<<<grid, kThreads, smem, s>>>(tA, tA2, tB, g, ea);
  e = cudaGetLastError();
  timing_end(c, name, s, ev);
  return e;
}

}  // namespace

cudaError_t launch_gemm12(rkv_ctx* c, const PassPlan& p, const int32_t* plan, cudaStream_t s) {
  const Dims& d = c->d;
  const int rows = p.n_rows;                    // dense rows
  GemmShape g{};
  if (d.mean_pre) {
    g.m_tiles = (rows + kTileM - 1) / kTileM;
    g.n_tiles = (2 * d.dff) / kEncN;
    g.nkb = d.dkv / kTileK;
    g.b_kwrap = g.nkb;
    g.status = c->status;
    const int zero_row = (d.B * d.R_cap + kTileM - 1) / kTileM * kTileM;   // past the tiles
    Epi12RArgs ea{c->H, d.dff, rows, plan + (p.dense ? p.off_d_dst : p.off_q_dst),
                  c->st.ref_idx, d.topk, d.R_cap, d.T_cap, c->P, zero_row};
    const CUtensorMap& tA = p.dense ? c->tm_qd128 : c->tm_qa128;
    return run_gemm<kEncN, 4, Epi12R>(c, tA, tA, c->tm_w12, g, ea, "rkv_gemm12_refpre_kernel", s);
  }
  g.m_tiles = (rows + kTileM / 2 - 1) / (kTileM / 2);
  g.n_tiles = (2 * d.dff) / kEncN;
  g.nkb = d.dkv / kTileK;
  g.b_kwrap = g.nkb;
  g.status = c->status;
  Epi12Args ea{c->H, d.dff, rows};
  return run_gemm<kEncN, 4, Epi12>(c, p.dense ? c->tm_qd : c->tm_qa, c->tm_m, c->tm_w12, g, ea,
                                   "rkv_gemm12_swiglu_kernel", s);
}

cudaError_t launch_pool_preact(rkv_ctx* c, const int32_t* tiles, int n_tiles, cudaStream_t s) {
  const Dims& d = c->d;
  GemmShape g{};
  g.m_tiles = n_tiles;
  g.n_tiles = (2 * d.dff) / kEncN;
  g.nkb = d.dkv / kTileK;
  g.b_kwrap = g.nkb;
  g.status = c->status;
  g.m_list = tiles;
  EpiPArgs ea{c->P, (int64_t)d.B * d.R_cap, 2 * d.dff};
  return run_gemm<kEncN, 4, EpiP>(c, c->tm_pool128, c->tm_pool128, c->tm_w12, g, ea,
                                  "rkv_pool_preact_kernel", s);
}

cudaError_t launch_gemm3_quant(rkv_ctx* c, const PassPlan& p, const int32_t* plan,
                               cudaStream_t s) {
  const Dims& d = c->d;
  GemmShape g{};
  g.m_tiles = (p.n_rows + kTileM - 1) / kTileM;  // dense rows
  g.nkb = (2 * d.dff) / kTileK;
  g.b_kwrap = d.dff / kTileK;
  g.status = c->status;
  Epi3Args ea{plan + (p.dense ? p.off_d_dst : p.off_q_dst), p.n_rows,
              static_cast<uint8_t*>(c->st.codes), static_cast<uint32_t*>(c->st.meta),
              d.code_bytes, d.G, d.bits, 0};
  const char* name = "rkv_gemm3_quant_kernel";
  // Tile width: the one whose whole waves of one-tile-per-SM finish first (a tile's
  // main loop costs in proportion to its width).
  auto waves = [&](int bn) {
    const int64_t tiles = (int64_t)g.m_tiles * (d.dc / bn);
    return ((tiles + c->num_sms - 1) / c->num_sms) * bn;
  };
  if (d.dc % 256 == 0 && waves(256) <= waves(128)) {
    g.n_tiles = d.dc / 256;
    ea.BN = 256;
    return run_gemm<256, 4, Epi3>(c, c->tm_h3, c->tm_h3, c->tm_w3, g, ea, name, s);
  }
  if (d.dc % 128 == 0) {
    g.n_tiles = d.dc / 128;
    ea.BN = 128;
    return run_gemm<128, 6, Epi3>(c, c->tm_h3, c->tm_h3,
                                  d.dc % 256 == 0 ? c->tm_w3_128 : c->tm_w3, g, ea, name, s);
  }
  g.n_tiles = d.dc / 64;
  ea.BN = 64;
  return run_gemm<64, 6, Epi3>(c, c->tm_h3, c->tm_h3, c->tm_w3, g, ea, name, s);
}

}  // namespace rkv
