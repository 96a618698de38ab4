// k_elementwise.cu - the memory-bound kernels of the codec: storage initialisation,
// weight repacking, reference-pool append (FP8 storage), query preparation for the
// tensor-core retrieval, and the reference-mean rows of the encoder operand.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include <climits>

#include "ptx.cuh"
#include "rkv_internal.h"

namespace rkv {
namespace {

__device__ __forceinline__ float fp8_to_float(uint8_t b) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
  return __half2float(__half(h));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat16 lo = __float2bfloat16_rn(a), hi = __float2bfloat16_rn(b);
  return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}

// ---------------------------------------------------------------- init
__global__ void init_storage_kernel(int32_t* pool_pos, int64_t n_pool, int32_t* ref_idx,
                                    int64_t n_idx) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_pool;
       i += (int64_t)gridDim.x * blockDim.x)
    pool_pos[i] = INT_MAX;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_idx;
       i += (int64_t)gridDim.x * blockDim.x)
    ref_idx[i] = -1;
}

// out[r][k] = src[k][col(r)] for a [K, N] row-major source; the W_c1/W_c2 pair is
// interleaved in 256-row tiles (128 rows of each) so one accumulator tile holds
// matching gate and value columns.
__global__ void repack_kernel(const __nv_bfloat16* __restrict__ a, const __nv_bfloat16* __restrict__ b,
                              __nv_bfloat16* __restrict__ out, int K, int N_src, int rows,
                              int interleave) {
  const int64_t total = (int64_t)rows * K;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / K);
    const int k = (int)(i % K);
    const __nv_bfloat16* src = a;
    int col = r;
    if (interleave) {
      const int j = r / kEncN, u = r % kEncN;
      col = j * (kEncN / 2) + (u % (kEncN / 2));
      src = (u < kEncN / 2) ? a : b;
    }
    out[i] = src[(int64_t)k * N_src + col];
  }
}

// ---------------------------------------------------------------- pool append
// One warp per reference row (plan row: {src row, pool row, pos, token row}).  Lane l
// takes the 8-element pieces e = (32 u + l) * 8: all of its loads are issued before any
// conversion, and the FP8 and bf16 stores of a warp cover whole contiguous segments.
// The squared norm of the FP8 row is summed exactly in integers: every E4M3 value is
// k * 2^-9 with |k| <= 448 * 2^9 < 2^18, so the row's sum of k^2 fits in int64 (2^36 per
// square); it is rounded to fp32 once and scaled by 2^-18 (exact), the correctly
// rounded squared norm.  (The float64 pipe would do the same, far more slowly.)
template <bool F32>
__global__ void __launch_bounds__(256)
    pool_append_kernel(const void* __restrict__ kv, int64_t stride,
                       const int32_t* __restrict__ plan, int n, int dkv, int R_cap,
                       uint8_t* __restrict__ pool8, __nv_bfloat16* __restrict__ poolb,
                       float* __restrict__ norm2, int32_t* __restrict__ pool_pos,
                       int32_t* __restrict__ ref_idx, int topk, uint8_t* __restrict__ codes,
                       int code_bytes, uint32_t* __restrict__ meta, int G) {
  constexpr int kPieces = F32 ? 4 : 8;          // pieces per lane in flight (32 registers)
  constexpr int kWords = F32 ? 2 : 1;           // 16-byte words per piece
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= n) return;
  const int64_t src = plan[4 * r + 0];
  const int64_t prow = plan[4 * r + 1];
  const int32_t pos = plan[4 * r + 2];
  const int64_t tok = plan[4 * r + 3];
  const uint4* in = reinterpret_cast<const uint4*>(
      static_cast<const uint8_t*>(kv) + src * stride * (F32 ? 4 : 2));
  long long acc = 0;
  for (int u0 = 0; u0 * 256 < dkv; u0 += kPieces) {
    uint4 raw[kPieces][kWords];
#pragma unroll
    for (int u = 0; u < kPieces; ++u) {
      const int e = ((u0 + u) * 32 + lane) * 8;
      if (e < dkv) {
#pragma unroll
        for (int w = 0; w < kWords; ++w) raw[u][w] = in[e / (8 / kWords) + w];
      }
    }
#pragma unroll
    for (int u = 0; u < kPieces; ++u) {
      const int e = ((u0 + u) * 32 + lane) * 8;
      if (e >= dkv) continue;
      float v[8];
      if (F32) {
#pragma unroll
        for (int w = 0; w < kWords; ++w) {
          v[4 * w] = __uint_as_float(raw[u][w].x), v[4 * w + 1] = __uint_as_float(raw[u][w].y);
          v[4 * w + 2] = __uint_as_float(raw[u][w].z), v[4 * w + 3] = __uint_as_float(raw[u][w].w);
        }
      } else {
        const uint32_t x[4] = {raw[u][0].x, raw[u][0].y, raw[u][0].z, raw[u][0].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[2 * i] = __uint_as_float(x[i] << 16);
          v[2 * i + 1] = __uint_as_float(x[i] & 0xFFFF0000u);
        }
      }
      uint32_t packed[2] = {0u, 0u};
      float d[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const __nv_fp8_storage_t q = __nv_cvt_float_to_fp8(v[i], __NV_SATFINITE, __NV_E4M3);
        packed[i >> 2] |= static_cast<uint32_t>(q) << (8 * (i & 3));
        d[i] = fp8_to_float(q);
        const int k = __float2int_rz(d[i] * 512.0f);   // exact: d = k * 2^-9
        acc += (long long)k * k;
      }
      *reinterpret_cast<uint2*>(pool8 + prow * dkv + e) = make_uint2(packed[0], packed[1]);
      *reinterpret_cast<uint4*>(poolb + prow * dkv + e) =
          make_uint4(pack_bf16x2(d[0], d[1]), pack_bf16x2(d[2], d[3]), pack_bf16x2(d[4], d[5]),
                     pack_bf16x2(d[6], d[7]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) {
    norm2[prow] = __ll2float_rn(acc) * 0x1p-18f;
    pool_pos[prow] = pos;
  }
  // the reference token's own entry: itself as the first reference, no code
  for (int t = lane; t < topk; t += 32) ref_idx[tok * topk + t] = t == 0 ? (int32_t)(prow % R_cap) : -1;
  for (int i = lane; i < code_bytes / 16; i += 32)
    reinterpret_cast<uint4*>(codes + tok * code_bytes)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = lane; i < G; i += 32) meta[tok * G + i] = 0u;
}

// ---------------------------------------------------------------- queries
// One block per retrieval-order row: bf16 copy of kv, or for fp32 kv the three bf16
// pieces hi, mid, lo with hi + mid + lo == x exactly (each piece takes the next 8
// significant bits), laid out [hi | mid | lo] along the row.
__global__ void prep_queries_kernel(const void* __restrict__ kv, int64_t stride, int kv_f32,
                                    const int32_t* __restrict__ q_src, int dkv, int parts,
                                    __nv_bfloat16* __restrict__ Q) {
  const int64_t row = blockIdx.x;
  const int64_t src = q_src[row];
  __nv_bfloat16* out = Q + row * (int64_t)parts * dkv;
  for (int e = threadIdx.x * 4; e < dkv; e += blockDim.x * 4) {
    if (src < 0) {
      for (int p = 0; p < parts; ++p)
        *reinterpret_cast<uint2*>(out + p * dkv + e) = make_uint2(0u, 0u);
      continue;
    }
    if (!kv_f32) {
      *reinterpret_cast<uint2*>(out + e) = *reinterpret_cast<const uint2*>(
          static_cast<const __nv_bfloat16*>(kv) + src * stride + e);
      continue;
    }
    const float4 x4 = *reinterpret_cast<const float4*>(
        static_cast<const float*>(kv) + src * stride + e);
    const float x[4] = {x4.x, x4.y, x4.z, x4.w};
    float pc[3][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float rem = x[i];
#pragma unroll
      for (int p = 0; p < 3; ++p) {
        const float h = __bfloat162float(__float2bfloat16_rn(rem));
        pc[p][i] = h;
        rem = __fsub_rn(rem, h);   // exact
      }
    }
    for (int p = 0; p < parts; ++p) {
      uint2 v;
      v.x = pack_bf16x2(pc[p][0], pc[p][1]);
      v.y = pack_bf16x2(pc[p][2], pc[p][3]);
      *reinterpret_cast<uint2*>(out + p * dkv + e) = v;
    }
  }
}

// bf16 kv rows: a plain copy into retrieval order.  One warp per row, each lane moving
// 16-byte pieces with eight loads in flight before the stores (the copy is bound by how
// many bytes are in flight, not by arithmetic).
__global__ void __launch_bounds__(256)
    prep_queries_bf16_kernel(const __nv_bfloat16* __restrict__ kv, int64_t stride,
                             const int32_t* __restrict__ q_src, int dkv, int m_pad,
                             __nv_bfloat16* __restrict__ Q) {
  const int lane = threadIdx.x & 31;
  const int pieces = dkv / 256;                       // 16-byte pieces per lane
  for (int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); row < m_pad;
       row += (int64_t)gridDim.x * 8) {
    const int64_t src = q_src[row];
    uint4* out = reinterpret_cast<uint4*>(Q + row * (int64_t)dkv);
    const uint4* in = reinterpret_cast<const uint4*>(kv + (src < 0 ? 0 : src) * stride);
    for (int p0 = 0; p0 < pieces; p0 += 8) {
      uint4 buf[8];
#pragma unroll
      for (int p = 0; p < 8; ++p)
        buf[p] = (src >= 0 && p0 + p < pieces) ? in[(p0 + p) * 32 + lane] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int p = 0; p < 8; ++p)
        if (p0 + p < pieces) out[(p0 + p) * 32 + lane] = buf[p];
    }
  }
}

// ---------------------------------------------------------------- mean rows
// One warp per dense row j (storage row d_dst[j]): M[j] = bf16(mean of the row's
// retrieved FP8 references).  The sum of at most four E4M3 values is exact in fp32; it
// is divided by k_i once, correctly rounded.  Each lane takes 8-element pieces
// e = (32 u + lane) * 8, four pieces in flight at a time.  (The row's kv operand is read
// by the encoder GEMM from the query rows, or from their dense copy.)
__global__ void __launch_bounds__(256)
    mean_rows_kernel(const int32_t* __restrict__ d_dst, const uint8_t* __restrict__ pool8,
                     const int32_t* __restrict__ ref_idx, int topk, int dkv, int T_cap,
                     int R_cap, int n_rows, __nv_bfloat16* __restrict__ M,
                     int* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  for (int64_t q = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); q < n_rows;
       q += (int64_t)gridDim.x * 8) {
    const int64_t dst = d_dst[q];
    __nv_bfloat16* xm = M + q * (int64_t)dkv;
    if (dst < 0) {
      for (int e = lane * 8; e < dkv; e += 256)
        *reinterpret_cast<uint4*>(xm + e) = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    const int64_t seq = dst / T_cap;
    const int32_t my = lane < topk ? ref_idx[dst * topk + lane] : -1;
    int64_t prow[4];
    bool ok[4];
    int k_i = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int32_t sl = __shfl_sync(0xffffffffu, my, t);
      ok[t] = t < topk && sl >= 0 && sl < R_cap;
      prow[t] = ok[t] ? seq * R_cap + sl : 0;
      k_i += ok[t] ? 1 : 0;
    }
    if (k_i == 0 && lane == 0) atomicOr(status, RKV_FLAG_UNWRITTEN);
    // the sum divided by k_i, correctly rounded: a multiply by the exact reciprocal for
    // k_i = 1, 2, 4, and the FMA-corrected division for k_i = 3
    const float kinv = 1.0f / (float)(k_i == 2 ? 2 : (k_i == 4 ? 4 : 1));
    for (int e0 = 0; e0 < dkv; e0 += 4 * 256) {
      uint2 rv[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + (u * 32 + lane) * 8;
        if (e < dkv) {
#pragma unroll
          for (int t = 0; t < 4; ++t)
            rv[t][u] = ok[t] ? *reinterpret_cast<const uint2*>(pool8 + prow[t] * dkv + e)
                             : make_uint2(0u, 0u);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + (u * 32 + lane) * 8;
        if (e >= dkv) continue;
        // exact sums of the E4M3 values (in any order: at most four of them)
        float s8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          if (!ok[t]) continue;
          fp8x4_add(rv[t][u].x, s8[0], s8[1], s8[2], s8[3]);
          fp8x4_add(rv[t][u].y, s8[4], s8[5], s8[6], s8[7]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) s8[i] = k_i == 3 ? div3_rn(s8[i]) : __fmul_rn(s8[i], kinv);
        uint4 o;
        o.x = pack_bf16x2(s8[0], s8[1]);
        o.y = pack_bf16x2(s8[2], s8[3]);
        o.z = pack_bf16x2(s8[4], s8[5]);
        o.w = pack_bf16x2(s8[6], s8[7]);
        *reinterpret_cast<uint4*>(xm + e) = o;
      }
    }
  }
}

int grid_for(int64_t n, int threads, int cap) {
  int64_t g = (n + threads - 1) / threads;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return (int)g;
}

}  // namespace

cudaError_t launch_init_storage(rkv_ctx* c, cudaStream_t s, int seq) {
  int64_t n_pool = (int64_t)c->d.B * c->d.R_cap;
  int64_t n_idx = (int64_t)c->d.B * c->d.T_cap * c->d.topk;
  int32_t* pool_pos = c->st.pool_pos;
  int32_t* ref_idx = c->st.ref_idx;
  if (seq >= 0) {
    n_pool = c->d.R_cap;
    n_idx = (int64_t)c->d.T_cap * c->d.topk;
    pool_pos += (int64_t)seq * n_pool;
    ref_idx += (int64_t)seq * n_idx;
  }
  cudaEvent_t ev;
  timing_begin(c, "rkv_init_storage_kernel", s, &ev);
  init_storage_kernel<<<grid_for(n_idx > n_pool ? n_idx : n_pool, 256, 4096), 256, 0, s>>>(
      pool_pos, n_pool, ref_idx, n_idx);
  cudaError_t e = cudaGetLastError();
  timing_end(c, "rkv_init_storage_kernel", s, ev);
  return e;
}

cudaError_t launch_repack_weights(rkv_ctx* c, const __nv_bfloat16* Wc1, const __nv_bfloat16* Wc2,
                                  const __nv_bfloat16* Wc3, const __nv_bfloat16* Wd,
                                  cudaStream_t s) {
  const Dims& d = c->d;
  repack_kernel<<<grid_for((int64_t)2 * d.dff * d.dkv, 256, 8192), 256, 0, s>>>(
      Wc1, Wc2, c->w12, d.dkv, d.dff, 2 * d.dff, 1);
  repack_kernel<<<grid_for((int64_t)d.dc * d.dff, 256, 8192), 256, 0, s>>>(
      Wc3, nullptr, c->w3, d.dff, d.dc, d.dc, 0);
  repack_kernel<<<grid_for((int64_t)d.dkv * d.dc, 256, 8192), 256, 0, s>>>(
      Wd, nullptr, c->wd, d.dc, d.dkv, d.dkv, 0);
  return cudaGetLastError();
}

cudaError_t launch_pool_append(rkv_ctx* c, const void* kv, int64_t stride, const int32_t* plan,
                               int n, cudaStream_t s) {
  const Dims& d = c->d;
  cudaEvent_t ev;
  timing_begin(c, "rkv_pool_append_kernel", s, &ev);
  auto kern = d.kv_f32 ? pool_append_kernel<true> : pool_append_kernel<false>;
  kern<<<(n + 7) / 8, 256, 0, s>>>(kv, stride, plan, n, d.dkv, d.R_cap,
                                   static_cast<uint8_t*>(c->st.pool_fp8),
                                   c->pool_bf16, c->st.pool_norm2,
                                   c->st.pool_pos, c->st.ref_idx, d.topk,
                                   static_cast<uint8_t*>(c->st.codes), d.code_bytes,
                                   static_cast<uint32_t*>(c->st.meta), d.G);
  cudaError_t e = cudaGetLastError();
  timing_end(c, "rkv_pool_append_kernel", s, ev);
  return e;
}

cudaError_t launch_prep_queries(rkv_ctx* c, const void* kv, int64_t stride, const int32_t* q_src,
                                int m_pad, cudaStream_t s) {
  const Dims& d = c->d;
  cudaEvent_t ev;
  timing_begin(c, "rkv_prep_queries_kernel", s, &ev);
  if (d.kv_f32)
    prep_queries_kernel<<<m_pad, 256, 0, s>>>(kv, stride, d.kv_f32, q_src, d.dkv, d.parts, c->Q);
  else
    prep_queries_bf16_kernel<<<grid_for(m_pad, 8, 16 * c->num_sms), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(kv), stride, q_src, d.dkv, m_pad, c->Q);
  cudaError_t e = cudaGetLastError();
  timing_end(c, "rkv_prep_queries_kernel", s, ev);
  return e;
}

cudaError_t launch_prep_dense(rkv_ctx* c, const void* kv, int64_t stride, const int32_t* d_src,
                              int n, cudaStream_t s) {
  const Dims& d = c->d;
  cudaEvent_t ev;
  timing_begin(c, "rkv_prep_queries_kernel", s, &ev);
  if (d.kv_f32)   // the first of the three bf16 pieces is the bf16 rounding of kv
    prep_queries_kernel<<<n, 256, 0, s>>>(kv, stride, d.kv_f32, d_src, d.dkv, 1, c->Qd);
  else
    prep_queries_bf16_kernel<<<grid_for(n, 8, 16 * c->num_sms), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(kv), stride, d_src, d.dkv, n, c->Qd);
  cudaError_t e = cudaGetLastError();
  timing_end(c, "rkv_prep_queries_kernel", s, ev);
  return e;
}

cudaError_t launch_mean_rows(rkv_ctx* c, const PassPlan& p, const int32_t* plan, cudaStream_t s) {
  const Dims& d = c->d;
  cudaEvent_t ev;
  timing_begin(c, "rkv_mean_rows_kernel", s, &ev);
  // dense rows: with one group the retrieval order's first n_rows rows
  const int32_t* d_dst = plan + (p.dense ? p.off_d_dst : p.off_q_dst);
  mean_rows_kernel<<<grid_for(p.n_rows, 8, 16 * c->num_sms), 256, 0, s>>>(
      d_dst, static_cast<const uint8_t*>(c->st.pool_fp8), c->st.ref_idx, d.topk,
      d.dkv, d.T_cap, d.R_cap, p.n_rows, c->M, c->status);
  cudaError_t e = cudaGetLastError();
  timing_end(c, "rkv_mean_rows_kernel", s, ev);
  return e;
}

// One block whose wait is never satisfied: the same bounded mbarrier wait as every
// pipeline here, so it must expire (about a second), raise RKV_FLAG_TIMEOUT and return.
// Exercises the failure-detection path without faulting or hanging the GPU.
__global__ void timeout_probe_kernel(int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, &abort_flag, status);  // nothing arrives
  __syncthreads();
}

cudaError_t launch_timeout_probe(rkv_ctx* c, cudaStream_t s) {
  timeout_probe_kernel<<<1, 32, 0, s>>>(c->status);
  return cudaGetLastError();
}

}  // namespace rkv
