// k_reconstruct.cu - fused read path (ResidualKV notes §2.5 boxed equation
// KV_hat = f_d(z~) + mean with f_d(z) = z W_d; §2.4 z~ = q Delta + min; §2.1 the
// restored pre-RoPE key is rotated at the token's own position; §2.7 only the selected
// tokens are restored).
//
// Work unit = (tile of 128 selected tokens, 256 output columns).  A CTA owns a
// contiguous range of units, so consecutive units mostly share the token tile:
//   1. the 128 epilogue threads gather the tile's codes and FP16 extremes (coalesced,
//      one 8-coordinate chunk per thread and step), dequantise them in fp32
//      (z~ = q * Delta + min, Delta = (max - min) / (2^b - 1)) and write bf16 z~ into
//      shared memory in the 128-byte-swizzled K-major layout the tensor core reads;
//   2. a TMA ring streams W_d^T tiles, one thread issues tcgen05.mma into a TMEM
//      accumulator (two accumulators alternate so the epilogue overlaps the next MMA);
//   3. the thread owning token row i reads its accumulator row, adds the mean of its
//      <= 4 FP8 references (exact fp32 sum, one division by k_i), rotates K columns
//      with RoPE (rotate-half pairs, cos/sin from float64-built tables combined by the
//      angle-addition formula) and stores K or V.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "tc_common.cuh"

namespace rkv {
namespace {

struct ReconArgs {
  const int32_t* seq;
  const int32_t* pos;
  int n_sel;
  int n_tiles;   // 2d_k / 256
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

constexpr uint32_t kBBytes = kDecN * 128;
constexpr uint32_t kTmemCols = 2 * kDecN;

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat16 lo = __float2bfloat16_rn(a), hi = __float2bfloat16_rn(b);
  return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}

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

__global__ void __launch_bounds__(kThreads, 1)
    reconstruct_kernel(const __grid_constant__ CUtensorMap tmW, ReconArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int nkb = a.dc / kTileK;
  uint8_t* sA = smem;                                  // nkb x [128 rows x 128 B]
  uint8_t* sB = smem + nkb * kTileABytes;              // stages x [256 rows x 128 B]
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
      mbar_init(&tempty[b], 128);
    }
    mbar_init(afull, 128);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch(&tmW);
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
    if (elect_one()) {
      Ring ring;
      int issued[8];
      uint32_t issued_phase[8];
      for (int s = 0; s < 8; ++s) issued[s] = 0, issued_phase[s] = 0;
      bool ok = true;
      for (int u = u_begin; u < u_end && ok; ++u) {
        const int n = u % a.n_tiles;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[ring.stage], ring.phase ^ 1u, abort_flag, a.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[ring.stage], kBBytes);
          tma_load_2d(sB + ring.stage * kBBytes, &tmW, &full[ring.stage], kb * kTileK, n * kDecN);
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
    if (elect_one()) {
      constexpr uint32_t idesc = idesc_bf16_f32(kTileM, kDecN);
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
        const uint32_t d = tmem + acc * kDecN;
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
  } else if (warp >= kEpiWarp0) {
    const int et = threadIdx.x - kEpiWarp0 * 32;   // 0..127 = TMEM lane = tile row
    const int ew = warp - kEpiWarp0;
    const int levels = (1 << a.bits) - 1;
    const int cpr = a.dc / 8;                       // 8-coordinate chunks per row
    int acc = 0;
    uint32_t acc_phase = 0;
    int cur_m = -1;
    // this thread's row
    bool valid = false;
    int64_t my_dst = -1, my_seq = 0;
    int my_pos = 0, k_i = 0;
    int64_t prow[4] = {0, 0, 0, 0};
    for (int u = u_begin; u < u_end; ++u) {
      const int m = u / a.n_tiles, n = u % a.n_tiles;
      if (m != cur_m) {
        cur_m = m;
        // ---- row metadata of the new token tile
        const int64_t gi = (int64_t)m * kTileM + et;
        valid = false;
        k_i = 0;
        if (gi < a.n_sel) {
          const int s = a.seq[gi], p = a.pos[gi];
          if (s < 0 || s >= a.B || p < 0 || p >= a.T_cap) {
            atomicOr(a.status, RKV_FLAG_BAD_INDEX);
          } else {
            my_dst = (int64_t)s * a.T_cap + p;
            my_seq = s;
            my_pos = p;
            for (int t = 0; t < a.topk; ++t) {
              const int32_t sl = a.ref_idx[my_dst * a.topk + t];
              if (sl >= 0 && sl < a.R_cap) prow[k_i++] = my_seq * a.R_cap + sl;
              else if (sl >= a.R_cap) atomicOr(a.status, RKV_FLAG_BAD_SLOT);
            }
            const int32_t s0 = a.ref_idx[my_dst * a.topk];
            if (s0 < 0) atomicOr(a.status, RKV_FLAG_UNWRITTEN);
            valid = (s0 >= 0 && s0 < a.R_cap) && k_i > 0;
          }
        }
        // ---- cooperative dequantisation of the 128 x d_c tile into swizzled smem.
        // Each item derives its row's storage index itself (no barrier among the
        // epilogue warps, so an aborted warp can never strand the others).
        for (int item = et; item < kTileM * cpr; item += 128) {
          const int r = item / cpr, ch = item % cpr;
          const int64_t ri = (int64_t)m * kTileM + r;
          int64_t dst = -1;
          if (ri < a.n_sel) {
            const int s = a.seq[ri], p = a.pos[ri];
            if (s >= 0 && s < a.B && p >= 0 && p < a.T_cap) {
              const int64_t dd = (int64_t)s * a.T_cap + p;
              const int32_t s0 = a.ref_idx[dd * a.topk];
              if (s0 >= 0 && s0 < a.R_cap) dst = dd;
            }
          }
          uint32_t w[4] = {0u, 0u, 0u, 0u};
          if (dst >= 0) {
            if (a.bits == 16) {
              const uint4 v = *reinterpret_cast<const uint4*>(a.codes + dst * a.code_bytes + ch * 16);
              w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
            } else {
              const uint32_t mt = a.meta[dst * a.G + (ch >> 2)];
              const float lo = __half2float(__ushort_as_half((unsigned short)(mt & 0xFFFFu)));
              const float hi = __half2float(__ushort_as_half((unsigned short)(mt >> 16)));
              const float delta = __fdiv_rn(__fsub_rn(hi, lo), (float)levels);
              uint32_t q;
              if (a.bits == 4)
                q = *reinterpret_cast<const uint32_t*>(a.codes + dst * a.code_bytes + ch * 4);
              else
                q = *reinterpret_cast<const uint16_t*>(a.codes + dst * a.code_bytes + ch * 2);
              float zt[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const uint32_t qi = (a.bits == 4) ? ((q >> (4 * i)) & 15u) : ((q >> (2 * i)) & 3u);
                zt[i] = __fadd_rn(__fmul_rn((float)qi, delta), lo);
              }
#pragma unroll
              for (int i = 0; i < 4; ++i) w[i] = pack_bf16x2(zt[2 * i], zt[2 * i + 1]);
            }
          }
          uint8_t* dstp = sA + (ch >> 3) * kTileABytes + sw128_offset(r, ch & 7);
          *reinterpret_cast<uint4*>(dstp) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(afull);
      }
      // ---- wait for this unit's accumulator
      if (!warp_wait(&tfull[acc], acc_phase, abort_flag, a.status)) break;
      tc_fence_after();
      const uint32_t tacc = tmem + ((uint32_t)(ew * 32) << 16) + (uint32_t)(acc * kDecN);
      const int64_t gi = (int64_t)m * kTileM + et;
      const int half = a.D / 2;
      const float kf = (float)(k_i > 0 ? k_i : 1);
      for (int hh = 0; hh < kDecN / a.D; ++hh) {
        const int c0 = n * kDecN + hh * a.D;      // first KV_hat column of this head
        const bool is_k = c0 < a.dk;
        void* out = is_k ? a.k_out : a.v_out;
        const int64_t out_col = (int64_t)(is_k ? c0 : c0 - a.dk);
        for (int pc = 0; pc < half; pc += 16) {
          const int xc = hh * a.D + pc;            // tile-local columns
          uint32_t xr[16], yr[16];
          tmem_ld16(tacc + xc, xr);
          tmem_ld16(tacc + xc + half, yr);
          tmem_ld_wait();
          if (gi >= a.n_sel) continue;
          float x[16], y[16];
          if (!valid) {
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = 0.f, y[i] = 0.f;
          } else {
            float mx[16], my[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) mx[i] = 0.f, my[i] = 0.f;
            for (int t = 0; t < k_i; ++t) {
              const uint8_t* rp = a.pool8 + prow[t] * a.dkv + c0 + pc;
              fp8x16_add(*reinterpret_cast<const uint4*>(rp), mx);
              fp8x16_add(*reinterpret_cast<const uint4*>(rp + half), my);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              x[i] = __fadd_rn(__uint_as_float(xr[i]), __fdiv_rn(mx[i], kf));
              y[i] = __fadd_rn(__uint_as_float(yr[i]), __fdiv_rn(my[i], kf));
            }
            if (is_k) {
              const float2* th = a.rope_hi + (int64_t)(my_pos >> 9) * half + pc;
              const float2* tl = a.rope_lo + (int64_t)(my_pos & (kRopeLo - 1)) * half + pc;
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float2 h2 = __ldg(th + i), l2 = __ldg(tl + i);
                const float cs = h2.x * l2.x - h2.y * l2.y;   // cos(A + B)
                const float sn = h2.y * l2.x + h2.x * l2.y;   // sin(A + B)
                const float xv = x[i], yv = y[i];
                x[i] = xv * cs - yv * sn;
                y[i] = yv * cs + xv * sn;
              }
            }
          }
          const int64_t rowoff = gi * (int64_t)a.dk + out_col + pc;
          store16(out, rowoff, x, a.out_f32);
          store16(out, rowoff + half, y, a.out_f32);
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
  if (warp == 2) {
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
  if (stages > 4) stages = 4;
  if (stages < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = fixed + (size_t)stages * kBBytes;
  cudaError_t e = cudaFuncSetAttribute(reconstruct_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ReconArgs a;
  a.seq = seq;
  a.pos = pos;
  a.n_sel = n_sel;
  a.n_tiles = d.dkv / kDecN;
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
  reconstruct_kernel<<<grid, kThreads, smem, s>>>(c->tm_wd, a);
  e = cudaGetLastError();
  timing_end(c, "rkv_reconstruct_kernel", s, ev);
  return e;
}

}  // namespace rkv
