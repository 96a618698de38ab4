// k_reconstruct.cu - fused read path (ResidualKV notes §2.5 boxed equation
// KV_hat = f_d(z~) + mean with f_d(z) = z W_d; §2.4 z~ = q Delta + min; §2.1 the
// restored pre-RoPE key is rotated at the token's own position; §2.7 only the selected
// tokens are restored).
//
// Work unit = (tile of 128 selected tokens, 128 output columns = one head for D = 128,
// two for D = 64).  A CTA owns a contiguous range of units, so consecutive units share
// the token tile.  Two warpgroup pairs alternate units, each owning one TMEM
// accumulator, so two units' epilogues are in flight while the tensor core runs ahead.
// Per token tile, the 512 epilogue threads (four warpgroups; the threads of TMEM lane r
// own token row r):
//   1. gather the row's codes and FP16 extremes and dequantise them in fp32
//      (z~ = q * Delta + min, Delta = (max - min) / (2^b - 1)) into bf16 z~ in shared
//      memory, in the 128-byte-swizzled K-major layout the tensor core reads;
//   2. build the row's RoPE cos/sin for the group's 32 column pairs (float64-built
//      two-level tables, angle-addition in fp32) once, and park them in TMEM.
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
constexpr uint32_t kRopeCol = 2 * kNT;      // per-group cos/sin caches after the accumulators
constexpr int kMaxStages = 4;

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

// s[i] += value of FP8 byte i of v (16 bytes), s held as 8 packed fp32 pairs; exact in
// fp32 for <= 4 addends (their bits span 2^-9 .. 2^11).
__device__ __forceinline__ void fp8x16_add2(uint4 v, uint64_t* s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      __nv_fp8x2_storage_t pair = static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * j)) & 0xFFFFu);
      const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3)));
      s[2 * i + j] = f32x2_add(s[2 * i + j], f32x2_pack(f.x, f.y));
    }
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
  uint64_t* afree = afull + 1;                         // the MMAs of a token tile are done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(afree + 1);
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
      mbar_init(&tempty[b], 8);                        // the owning pair's eight warps
    }
    mbar_init(afull, kEpiGroups * 4);                   // one arrival per epilogue warp
    mbar_init(afree, 1);
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
          // the previous tile's A may be overwritten once its MMAs are done
          if (cur_m >= 0) umma_commit(afree);
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
    // [32 (w % 4), +32), so every group owns the same 128 rows.  Groups 2p and 2p+1 form
    // pair p, which handles the CTA's units of parity p with accumulator p; within a
    // unit, group 2p+h takes column pairs [32h, 32h+32) in two chunks of 16.  Every
    // group dequantises a quarter of each row's code groups.
    const int ew = warp & 3;
    const int wg = (warp - kEpiWarpR) >> 2;
    const int pr = wg >> 1, hw = wg & 1;
    const int row = ew * 32 + (int)lane_id();        // TMEM lane = tile row
    const uint32_t lane_base = (uint32_t)(ew * 32) << 16;
    const int levels = (1 << a.bits) - 1;
    const int P = a.D / 2;                           // pairs per head
    const int jbase = (32 * hw) % P;                 // first pair index of the group
    const uint32_t rope_col = kRopeCol + 64u * (uint32_t)wg;
    const int g0 = wg * a.G / kEpiGroups;            // this group's code groups [g0, g1)
    const int g_per = (wg + 1) * a.G / kEpiGroups - g0;
    uint32_t acc_phase = 0, afree_phase = 0;
    int cur_m = -1;
    bool valid = false;
    int k_i = 0;
    int32_t rrow[4] = {0, 0, 0, 0};                // pool rows of the references
    int my_pos = 0;
    bool have_next = false;
    int next_m = -1, next_s = -1, next_p = -1;
    bool ok = true;
    for (int u = u_begin; u < u_end && ok; ++u) {
      const int m = u / a.n_tiles, n = u % a.n_tiles;
      const int64_t gi = (int64_t)m * kTileM + row;
      if (m != cur_m) {
        // wait until the tensor core is done with the previous tile's A
        if (cur_m >= 0) {
          if (!warp_wait(afree, afree_phase, abort_flag, a.status)) break;
          afree_phase ^= 1u;
        }
        cur_m = m;
        // ---- this row's metadata (prefetched while the previous tile was processed)
        int s_, p_;
        if (have_next && next_m == m) {
          s_ = next_s;
          p_ = next_p;
        } else {
          s_ = gi < a.n_sel ? a.seq[gi] : -1;
          p_ = gi < a.n_sel ? a.pos[gi] : -1;
        }
        valid = false;
        k_i = 0;
        bool in_range = false;
        int64_t dst = 0;
        my_pos = 0;
        if (gi < a.n_sel) {
          if (s_ < 0 || s_ >= a.B || p_ < 0 || p_ >= a.T_cap) {
            if (wg == 0) atomicOr(a.status, RKV_FLAG_BAD_INDEX);
          } else {
            in_range = true;
            dst = (int64_t)s_ * a.T_cap + p_;
            my_pos = p_;
          }
        }
        // one round trip: slots, extremes and codes together
        int32_t sl[4] = {-1, -1, -1, -1};
        uint32_t mt[4] = {0u, 0u, 0u, 0u};
        uint4 cw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) cw[i] = make_uint4(0u, 0u, 0u, 0u);
        const uint8_t* crow = a.codes + dst * a.code_bytes;
        if (in_range) {
#pragma unroll
          for (int t = 0; t < 4; ++t)
            if (t < a.topk) sl[t] = a.ref_idx[dst * a.topk + t];
          if (a.bits != 16) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if (i < g_per) {
                const int g = g0 + i;
                mt[i] = a.meta[dst * a.G + g];
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
        // the next tile's row metadata, for the next tile change
        have_next = false;
        {
          const int u_next = (m + 1) * a.n_tiles;
          if (u_next < u_end) {
            const int64_t gn = (int64_t)(m + 1) * kTileM + row;
            next_m = m + 1;
            next_s = gn < a.n_sel ? a.seq[gn] : -1;
            next_p = gn < a.n_sel ? a.pos[gn] : -1;
            have_next = true;
          }
        }
        if (in_range) {
          if (sl[0] < 0 && wg == 0) atomicOr(a.status, RKV_FLAG_UNWRITTEN);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            if (sl[t] >= a.R_cap && wg == 0) atomicOr(a.status, RKV_FLAG_BAD_SLOT);
            if (sl[t] >= 0 && sl[t] < a.R_cap) {
              const int32_t q = s_ * a.R_cap + sl[t];
              if (k_i == 0) rrow[0] = q;
              else if (k_i == 1) rrow[1] = q;
              else if (k_i == 2) rrow[2] = q;
              else rrow[3] = q;
              ++k_i;
            }
          }
          valid = (sl[0] >= 0 && sl[0] < a.R_cap) && k_i > 0;
        }
        // ---- dequantise this row's share of code groups into the swizzled A tile
        if (a.bits == 16) {
          for (int g = g0; g < g0 + g_per; ++g) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int ch = g * 4 + q;
              const uint4 v = valid ? reinterpret_cast<const uint4*>(crow + (int64_t)g * 64)[q]
                                    : make_uint4(0u, 0u, 0u, 0u);
              *reinterpret_cast<uint4*>(sA + (ch >> 3) * kTileABytes + sw128_offset(row, ch & 7)) = v;
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (i >= g_per) break;
            const int g = g0 + i;
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
        // A is ready for the tensor core (each thread publishes its shared-memory writes
        // to the async proxy; one lane per warp arrives); the RoPE cache below is only
        // needed later
        fence_proxy_async_smem();
        __syncwarp();
        if (lane_id() == 0) mbar_arrive(afull);
        // ---- cos/sin of the group's 32 pairs at the row's own position, into TMEM
        {
          const float4* th = reinterpret_cast<const float4*>(a.rope_hi + (int64_t)(my_pos >> 9) * P + jbase);
          const float4* tl = reinterpret_cast<const float4*>(a.rope_lo + (int64_t)(my_pos & (kRopeLo - 1)) * P + jbase);
#pragma unroll 1
          for (int hb = 0; hb < 4; ++hb) {             // 8 pairs at a time
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
      }
      if (((u - u_begin) & 1) != pr) continue;         // the other pair's unit
      // ---- this group's 32 pairs of the unit, 16 at a time
      bool have_acc = false;
      const uint32_t tacc = tmem + lane_base + (uint32_t)(pr * kNT);
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        const int slot = 32 * hw + 16 * c;             // pair slot within the unit
        const int hl = slot / P, j0 = slot % P;        // head within the unit, first pair
        const int xcol = hl * a.D + j0, ycol = xcol + P;
        const int c0 = n * kNT + hl * a.D;             // first KV_hat column of the head
        const bool is_k = c0 < a.dk;
        // mean of the references first (no TMEM dependency)
        uint64_t mx2[8], my2[8];                        // packed fp32 pairs
#pragma unroll
        for (int i = 0; i < 8; ++i) mx2[i] = 0ull, my2[i] = 0ull;
        if (valid) {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            if (t < k_i) {
              const uint8_t* rp = a.pool8 + (int64_t)rrow[t] * a.dkv + c0 + j0;
              const uint4 rx = __ldg(reinterpret_cast<const uint4*>(rp));
              const uint4 ry = __ldg(reinterpret_cast<const uint4*>(rp + P));
              fp8x16_add2(rx, mx2);
              fp8x16_add2(ry, my2);
            }
          }
        }
        float mx[16], my[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          f32x2_unpack(mx2[i], mx[2 * i], mx[2 * i + 1]);
          f32x2_unpack(my2[i], my[2 * i], my[2 * i + 1]);
        }
        if (valid) {
          if (k_i == 3) {
#pragma unroll
            for (int i = 0; i < 16; ++i) mx[i] = __fdiv_rn(mx[i], 3.0f), my[i] = __fdiv_rn(my[i], 3.0f);
          } else {
            const float kinv = 1.0f / (float)k_i;     // exact for k_i = 1, 2, 4
#pragma unroll
            for (int i = 0; i < 16; ++i) mx[i] = __fmul_rn(mx[i], kinv), my[i] = __fmul_rn(my[i], kinv);
          }
        }
        if (!have_acc) {
          if (!warp_wait(&tfull[pr], acc_phase, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          have_acc = true;
        }
        {
          uint32_t xr[16], yr[16];
          tmem_ld16(tacc + xcol, xr);
          tmem_ld16(tacc + ycol, yr);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            mx[i] = __fadd_rn(__uint_as_float(xr[i]), mx[i]);
            my[i] = __fadd_rn(__uint_as_float(yr[i]), my[i]);
          }
        }
        if (is_k) {
          uint32_t cs[32];
          tmem_ld32(tmem + lane_base + rope_col + 32u * c, cs);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float cc = __uint_as_float(cs[2 * i]), sn = __uint_as_float(cs[2 * i + 1]);
            const float xv = mx[i], yv = my[i];
            mx[i] = xv * cc - yv * sn;
            my[i] = yv * cc + xv * sn;
          }
        }
        if (!valid) {
#pragma unroll
          for (int i = 0; i < 16; ++i) mx[i] = 0.f, my[i] = 0.f;
        }
        if (gi < a.n_sel) {
          void* out = is_k ? a.k_out : a.v_out;
          const int64_t rowoff = gi * (int64_t)a.dk + (is_k ? c0 : c0 - a.dk) + j0;
          if (a.out_f32) {
            float* o = static_cast<float*>(out) + rowoff;
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
            __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out) + rowoff;
            st_global_v8(o, wx);                        // 16 bf16 = one 32-byte sector
            st_global_v8(o + P, wy);
          }
        }
      }
      if (!ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane_id() == 0) mbar_arrive(&tempty[pr]);
      acc_phase ^= 1u;
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
