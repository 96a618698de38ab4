// k_reconstruct.cu - fused read path (ResidualKV notes §2.5 boxed equation
// KV_hat = f_d(z~) + mean with f_d(z) = z W_d; §2.4 z~ = q Delta + min; §2.1 the
// restored pre-RoPE key is rotated at the token's own position; §2.7 only the selected
// tokens are restored).
//
// Work unit = (tile of 128 selected tokens, 128 output columns = one head for D = 128,
// two for D = 64).  A CTA owns a contiguous range of units, so consecutive units share
// the token tile.  Per token tile, the 512 epilogue threads (four warpgroups; the
// threads of TMEM lane r own token row r):
//   1. gather the row's codes and FP16 extremes and dequantise them in fp32
//      (z~ = q * Delta + min, Delta = (max - min) / (2^b - 1)) into bf16 z~ in shared
//      memory, in the 128-byte-swizzled K-major layout the tensor core reads;
//   2. build the row's RoPE cos/sin for its 16 column pairs (float64-built two-level
//      tables, angle-addition in fp32) once, and park them in spare TMEM columns.
// Per unit, a TMA ring streams W_d^T tiles, one thread issues tcgen05.mma into one of
// two TMEM accumulators, and each epilogue thread reads its accumulator row, adds the
// mean of its <= 4 FP8 references (exact fp32 sum, one division by k_i; every gather
// is a whole 32-byte sector), rotates K columns with the cached cos/sin and stores K
// or V in whole sectors.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "tc_common.cuh"

namespace rkv {
namespace {

// 20 warps: TMA + TMEM, MMA, two idle, 4 x 4 epilogue.  The register file is split
// over the four SM sub-partitions, so 18 or 20 warps both cap a thread at 96 registers.
constexpr int kReconThreads = 640;
constexpr int kEpiGroups = 4;
constexpr int kEpiWarpR = 4;               // first epilogue warp
constexpr int kNT = 128;                    // output columns per unit
constexpr uint32_t kBBytes = kNT * 128;     // one 64-wide k-block of W_d^T rows
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kRopeCol = 2 * kNT;      // cos/sin cache after the two accumulators
constexpr int kMaxStages = 6;

struct ReconArgs {
  const int32_t* seq;
  const int32_t* pos;
  int n_sel;
  int n_tiles;   // 2d_k / 128
  int units;
  int stages;
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
  int* status;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat16 lo = __float2bfloat16_rn(a), hi = __float2bfloat16_rn(b);
  return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}

// s[i] += value of FP8 byte i of v (16 bytes); exact in fp32 for <= 4 addends.
__device__ __forceinline__ void fp8x16_add(uint4 v, float* s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      __nv_fp8x2_storage_t pair = static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * j)) & 0xFFFFu);
      float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3)));
      s[4 * i + 2 * j] = __fadd_rn(s[4 * i + 2 * j], f.x);
      s[4 * i + 2 * j + 1] = __fadd_rn(s[4 * i + 2 * j + 1], f.y);
    }
  }
}

__device__ __forceinline__ void store8(void* base, int64_t off, const float* v, int out_f32) {
  if (out_f32) {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
    d[0] = make_float4(v[0], v[1], v[2], v[3]);
    d[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + off) =
        make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                   pack_bf16x2(v[6], v[7]));
  }
}

__device__ __forceinline__ void store16(void* base, int64_t off, const float* v, int out_f32) {
  if (out_f32) {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
    uint4* d = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + off);
#pragma unroll
    for (int i = 0; i < 2; ++i)
      d[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                        pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
  }
}

__global__ void __launch_bounds__(kReconThreads, 1)
    reconstruct_kernel(const __grid_constant__ CUtensorMap tmW, ReconArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int nkb = a.dc / kTileK;
  uint8_t* sA = smem;                                  // nkb x [128 rows x 128 B]
  uint8_t* sB = smem + nkb * kTileABytes;              // stages x [128 rows x 128 B]
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + a.stages * kBBytes);
  uint64_t* empty = full + a.stages;
  uint64_t* tfull = empty + a.stages;
  uint64_t* tempty = tfull + 2;
  uint64_t* afull = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(afull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int u_begin = (int)(((int64_t)blockIdx.x * a.units) / gridDim.x);
  const int u_end = (int)(((int64_t)(blockIdx.x + 1) * a.units) / gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kEpiGroups * 128);
    }
    mbar_init(afull, kEpiGroups * 128);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch(&tmW);
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
      int issued[kMaxStages];
      uint32_t issued_phase[kMaxStages];
      for (int s = 0; s < kMaxStages; ++s) issued[s] = 0, issued_phase[s] = 0;
      bool ok = true;
      for (int u = u_begin; u < u_end && ok; ++u) {
        const int n = u % a.n_tiles;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[ring.stage], ring.phase ^ 1u, abort_flag, a.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[ring.stage], kBBytes);
          tma_load_2d(sB + ring.stage * kBBytes, &tmW, &full[ring.stage], kb * kTileK, n * kNT);
          issued[ring.stage] = 1;
          issued_phase[ring.stage] = ring.phase;
          ring.next(a.stages);
        }
      }
      if (!ok)
        for (int s = 0; s < a.stages; ++s)
          if (issued[s]) drain_wait(&full[s], issued_phase[s]);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t idesc = idesc_bf16_f32(kTileM, kNT);
      Ring ring;
      int acc = 0;
      uint32_t acc_phase = 0, a_phase = 0;
      int cur_m = -1;
      bool ok = true, any = false;
      int last_stage = 0;
      uint32_t last_phase = 0;
      for (int u = u_begin; u < u_end && ok; ++u) {
        const int m = u / a.n_tiles;
        if (m != cur_m) {
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
          const uint32_t a0 = smem_u32(sA + kb * kTileABytes);
          const uint32_t b0 = smem_u32(sB + ring.stage * kBBytes);
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k)
            umma_bf16(d, sdesc_sw128(a0 + k * 32), sdesc_sw128(b0 + k * 32), idesc,
                      (kb | k) != 0 ? 1u : 0u);
          umma_commit(&empty[ring.stage]);
          any = true;
          last_stage = ring.stage;
          last_phase = ring.phase;
          ring.next(a.stages);
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
  } else if (warp >= kEpiWarpR) {
    // Four groups of four consecutive warps (warps 4..19).  Warp w reads TMEM lanes
    // [32 (w % 4), +32), so every group owns the same 128 rows; group g takes 16 of
    // each unit's 64 column pairs and a quarter of each row's code groups.
    const int ew = warp & 3;
    const int wg = (warp - kEpiWarpR) >> 2;
    const int row = ew * 32 + (int)lane_id();        // TMEM lane = tile row
    const uint32_t lane_base = (uint32_t)(ew * 32) << 16;
    const int levels = (1 << a.bits) - 1;
    const int P = a.D / 2;                           // pairs per head
    const int slot0 = 16 * wg;                       // first of this group's 16 pair slots
    const int hl = slot0 / P, j0 = slot0 % P;        // head within the unit, first pair
    const int xcol = hl * a.D + j0;                  // tile-local columns of x and y
    const int ycol = xcol + P;
    const uint32_t rope_col = kRopeCol + 32u * (uint32_t)wg;
    const int g0 = wg * a.G / kEpiGroups;            // this group's code groups [g0, g1)
    const int g_per = (wg + 1) * a.G / kEpiGroups - g0;
    int acc = 0;
    uint32_t acc_phase = 0;
    int cur_m = -1;
    bool valid = false;
    int k_i = 0;
    int32_t rrow[4] = {0, 0, 0, 0};                // pool rows of the references
    for (int u = u_begin; u < u_end; ++u) {
      const int m = u / a.n_tiles, n = u % a.n_tiles;
      const int64_t gi = (int64_t)m * kTileM + row;
      if (m != cur_m) {
        cur_m = m;
        // ---- this row's metadata
        valid = false;
        k_i = 0;
        int64_t dst = 0;
        int my_pos = 0;
        if (gi < a.n_sel) {
          const int s = a.seq[gi], p = a.pos[gi];
          if (s < 0 || s >= a.B || p < 0 || p >= a.T_cap) {
            if (wg == 0) atomicOr(a.status, RKV_FLAG_BAD_INDEX);
          } else {
            dst = (int64_t)s * a.T_cap + p;
            my_pos = p;
            int32_t sl[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) sl[t] = t < a.topk ? a.ref_idx[dst * a.topk + t] : -1;
            if (sl[0] < 0 && wg == 0) atomicOr(a.status, RKV_FLAG_UNWRITTEN);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              if (sl[t] >= a.R_cap && wg == 0) atomicOr(a.status, RKV_FLAG_BAD_SLOT);
              if (sl[t] >= 0 && sl[t] < a.R_cap) {
                const int32_t q = s * a.R_cap + sl[t];
                if (k_i == 0) rrow[0] = q;
                else if (k_i == 1) rrow[1] = q;
                else if (k_i == 2) rrow[2] = q;
                else rrow[3] = q;
                ++k_i;
              }
            }
            valid = (sl[0] >= 0 && sl[0] < a.R_cap) && k_i > 0;
          }
        }
        // ---- dequantise this row's share of code groups into the swizzled A tile
        const uint8_t* crow = a.codes + (valid ? dst : 0) * a.code_bytes;
        const uint32_t* mrow = a.meta + (valid ? dst : 0) * a.G;
        const int gstep = a.bits == 16 ? 1 : 2;
        for (int gb = 0; gb < g_per; gb += gstep) {
          const int ng = g_per - gb < gstep ? g_per - gb : gstep;
          uint32_t mt[4] = {0u, 0u, 0u, 0u};
          uint4 cw[4];
          // every load of the step's groups is issued before any is used
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            cw[i] = make_uint4(0u, 0u, 0u, 0u);
            if (!valid) continue;
            if (a.bits == 16) {           // one group = 64 bytes = four chunks
              cw[i] = reinterpret_cast<const uint4*>(crow + (int64_t)(g0 + gb) * 64)[i];
            } else if (i < ng) {
              const int g = g0 + gb + i;
              mt[i] = mrow[g];
              if (a.bits == 4) {
                cw[i] = *reinterpret_cast<const uint4*>(crow + (int64_t)g * 16);
              } else {
                const uint2 v = *reinterpret_cast<const uint2*>(crow + (int64_t)g * 8);
                cw[i] = make_uint4(v.x, v.y, 0u, 0u);
              }
            }
          }
          if (a.bits == 16) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int ch = (g0 + gb) * 4 + q;
              *reinterpret_cast<uint4*>(sA + (ch >> 3) * kTileABytes + sw128_offset(row, ch & 7)) = cw[q];
            }
            continue;
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (i >= ng) break;
            const int g = g0 + gb + i;
            const float lo = __half2float(__ushort_as_half((unsigned short)(mt[i] & 0xFFFFu)));
            const float hi = __half2float(__ushort_as_half((unsigned short)(mt[i] >> 16)));
            const float delta = __fdiv_rn(__fsub_rn(hi, lo), (float)levels);
            const uint32_t w4[4] = {cw[i].x, cw[i].y, cw[i].z, cw[i].w};
            // group g = coordinates [32g, 32g+32) = four 16-byte chunks of 8 values
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t o[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int k = 8 * q + 2 * e;           // first of two coordinates
                uint32_t q0, q1;
                if (a.bits == 4) {
                  q0 = (w4[k >> 3] >> (4 * (k & 7))) & 15u;
                  q1 = (w4[k >> 3] >> (4 * (k & 7) + 4)) & 15u;
                } else {
                  q0 = (w4[k >> 4] >> (2 * (k & 15))) & 3u;
                  q1 = (w4[k >> 4] >> (2 * (k & 15) + 2)) & 3u;
                }
                o[e] = valid ? pack_bf16x2(__fadd_rn(__fmul_rn((float)q0, delta), lo),
                                           __fadd_rn(__fmul_rn((float)q1, delta), lo))
                             : 0u;
              }
              const int ch = g * 4 + q;
              *reinterpret_cast<uint4*>(sA + (ch >> 3) * kTileABytes + sw128_offset(row, ch & 7)) =
                  make_uint4(o[0], o[1], o[2], o[3]);
            }
          }
        }
        // ---- cos/sin of this group's 32 pairs at the row's own position, into TMEM
        {
          const float4* th = reinterpret_cast<const float4*>(a.rope_hi + (int64_t)(my_pos >> 9) * P + j0);
          const float4* tl = reinterpret_cast<const float4*>(a.rope_lo + (int64_t)(my_pos & (kRopeLo - 1)) * P + j0);
#pragma unroll 1
          for (int hb = 0; hb < 2; ++hb) {             // 8 pairs at a time
            float4 hv[4], lv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) hv[i] = __ldg(th + 4 * hb + i), lv[i] = __ldg(tl + 4 * hb + i);
            uint32_t cs[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float hc = e ? hv[i].z : hv[i].x, hs = e ? hv[i].w : hv[i].y;
                const float lc = e ? lv[i].z : lv[i].x, ls = e ? lv[i].w : lv[i].y;
                cs[4 * i + 2 * e] = __float_as_uint(hc * lc - hs * ls);       // cos(A + B)
                cs[4 * i + 2 * e + 1] = __float_as_uint(hs * lc + hc * ls);   // sin(A + B)
              }
            }
            tmem_st16(tmem + lane_base + rope_col + 16u * hb, cs);
          }
          tmem_st_wait();
        }
        fence_proxy_async_smem();
        mbar_arrive(afull);
      }
      // ---- this unit's 16 pairs: mean of the references first (no TMEM dependency)
      const int c0 = n * kNT + hl * a.D;               // first KV_hat column of the head
      const bool is_k = c0 < a.dk;
      float mx[16], my[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) mx[i] = 0.f, my[i] = 0.f;
      if (valid) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          if (t < k_i) {
            const uint8_t* rp = a.pool8 + (int64_t)rrow[t] * a.dkv + c0 + j0;
            const uint4 rx = __ldg(reinterpret_cast<const uint4*>(rp));
            const uint4 ry = __ldg(reinterpret_cast<const uint4*>(rp + P));
            fp8x16_add(rx, mx);
            fp8x16_add(ry, my);
          }
        }
        if (k_i == 3) {
#pragma unroll
          for (int i = 0; i < 16; ++i) mx[i] = __fdiv_rn(mx[i], 3.0f), my[i] = __fdiv_rn(my[i], 3.0f);
        } else {
          const float kinv = 1.0f / (float)k_i;       // exact for k_i = 1, 2, 4
#pragma unroll
          for (int i = 0; i < 16; ++i) mx[i] = __fmul_rn(mx[i], kinv), my[i] = __fmul_rn(my[i], kinv);
        }
      }
      // ---- accumulator rows
      if (!warp_wait(&tfull[acc], acc_phase, abort_flag, a.status)) break;
      tc_fence_after();
      const uint32_t tacc = tmem + lane_base + (uint32_t)(acc * kNT);
      void* out = is_k ? a.k_out : a.v_out;
      const int64_t rowoff = gi * (int64_t)a.dk + (is_k ? c0 : c0 - a.dk) + j0;
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {                 // 8 pairs at a time
        uint32_t xr[8], yr[8], cs[16];
        tmem_ld8(tacc + xcol + 8 * hb, xr);
        tmem_ld8(tacc + ycol + 8 * hb, yr);
        if (is_k) tmem_ld16(tmem + lane_base + rope_col + 16u * hb, cs);
        tmem_ld_wait();
        float x[8], y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          x[i] = __fadd_rn(__uint_as_float(xr[i]), mx[8 * hb + i]);
          y[i] = __fadd_rn(__uint_as_float(yr[i]), my[8 * hb + i]);
        }
        if (is_k) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float c = __uint_as_float(cs[2 * i]), s = __uint_as_float(cs[2 * i + 1]);
            const float xv = x[i], yv = y[i];
            x[i] = xv * c - yv * s;
            y[i] = yv * c + xv * s;
          }
        }
        if (!valid) {
#pragma unroll
          for (int i = 0; i < 8; ++i) x[i] = 0.f, y[i] = 0.f;
        }
        if (gi < a.n_sel) {
          store8(out, rowoff + 8 * hb, x, a.out_f32);
          store8(out, rowoff + P + 8 * hb, y, a.out_f32);
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_reconstruct(rkv_ctx* c, const int32_t* seq, const int32_t* pos, int n_sel,
                               void* k_out, void* v_out, cudaStream_t s) {
  const Dims& d = c->d;
  if (n_sel <= 0) return cudaSuccess;
  const size_t fixed = 1024 + (size_t)(d.dc / kTileK) * kTileABytes + 256;
  int stages = (int)((232448 - fixed) / kBBytes);
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = fixed + (size_t)stages * kBBytes;
  cudaError_t e = cudaFuncSetAttribute(reconstruct_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ReconArgs a;
  a.seq = seq;
  a.pos = pos;
  a.n_sel = n_sel;
  a.n_tiles = d.dkv / kNT;
  const int m_tiles = (n_sel + kTileM - 1) / kTileM;
  a.units = m_tiles * a.n_tiles;
  a.stages = stages;
  a.codes = static_cast<const uint8_t*>(c->st.codes);
  a.meta = static_cast<const uint32_t*>(c->st.meta);
  a.ref_idx = c->st.ref_idx;
  a.pool8 = static_cast<const uint8_t*>(c->st.pool_fp8);
  a.rope_lo = c->rope_lo;
  a.rope_hi = c->rope_hi;
  a.k_out = k_out;
  a.v_out = v_out;
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
  a.status = c->status;
  const int grid = a.units < c->num_sms ? a.units : c->num_sms;
  cudaEvent_t ev;
  timing_begin(c, "rkv_reconstruct_kernel", s, &ev);
  reconstruct_kernel<<<grid, kReconThreads, smem, s>>>(c->tm_wd, a);
  e = cudaGetLastError();
  timing_end(c, "rkv_reconstruct_kernel", s, ev);
  return e;
}

}  // namespace rkv
