// k_attention.cu - sparse-layer attention over restored K/V (ResidualKV notes §2.7, the
// output equation o = softmax(q K_hat^T / sqrt(D)) V_hat over the selected tokens).
//
// Decode attention is a few dot products per token against K/V rows that a restore has
// just written (they are still in L2), so the work is split over the tokens, not over
// the heads: a CTA takes one chunk of selected tokens and one key/value head, scores
// the chunk against every query head of that head's group, and keeps a chunk-local
// softmax (its maximum m, its sum l of exp(s - m), and sum exp(s - m) v).  A second
// launch merges the chunks of each query head: M = max m_c, L = sum l_c e^(m_c - M),
// o = sum acc_c e^(m_c - M) / L.  Everything is fp32; exp is the library expf.
#include <cuda_bf16.h>
#include <stdint.h>

#include <cfloat>

#include "ptx.cuh"
#include "rkv_internal.h"

namespace rkv {
namespace {

constexpr int kAttnThreads = 256;

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  v = red[0];
  for (int i = 1; i < kAttnThreads / 32; ++i) v = fmaxf(v, red[i]);
  return v;
}

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  v = 0.f;
  for (int i = 0; i < kAttnThreads / 32; ++i) v += red[i];
  return v;
}

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* f) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void load8(const float* p, float* f) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w, f[4] = b.x, f[5] = b.y, f[6] = b.z, f[7] = b.w;
}

__device__ __forceinline__ float load1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float load1(const float* p) { return *p; }

// Grid (chunks, N).  Dynamic shared memory: q [G][D] (scaled by 1/sqrt(D)), then the
// scores / weights [G][chunk].  part_m, part_l: [chunks][Hq]; part_acc: [chunks][Hq][D].
template <typename T>
__global__ void __launch_bounds__(kAttnThreads)
    attn_partial_kernel(const float* __restrict__ q, const T* __restrict__ k,
                        const T* __restrict__ v, int n, int N, int D, int G, int chunk,
                        float* __restrict__ part_m, float* __restrict__ part_l,
                        float* __restrict__ part_acc) {
  extern __shared__ float sm[];
  __shared__ float red[kAttnThreads / 32];
  float* qs = sm;                     // [G][D]
  float* ss = sm + G * D;             // [G][chunk]
  const int c = blockIdx.x, g = blockIdx.y;
  const int Hq = G * N;
  const int j0 = c * chunk;
  const int cn = min(chunk, n - j0);
  const float scale = rsqrtf((float)D);
  for (int i = threadIdx.x; i < G * D; i += kAttnThreads)
    qs[i] = q[(size_t)(g * G + i / D) * D + (i % D)] * scale;
  __syncthreads();

  // scores: one token per thread, its whole row against every query head of the group
  for (int j = threadIdx.x; j < cn; j += kAttnThreads) {
    const T* kr = k + ((size_t)(j0 + j) * N + g) * D;
    float s[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) s[h] = 0.f;
    for (int d = 0; d < D; d += 8) {
      float kf[8];
      load8(kr + d, kf);
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        if (h < G) {
#pragma unroll
          for (int e = 0; e < 8; ++e) s[h] = fmaf(qs[h * D + d + e], kf[e], s[h]);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 8; ++h)
      if (h < G) ss[h * chunk + j] = s[h];
  }
  __syncthreads();

  // chunk-local softmax of each query head: m, weights exp(s - m), l
  for (int h = 0; h < G; ++h) {
    float mx = -FLT_MAX;
    for (int j = threadIdx.x; j < cn; j += kAttnThreads) mx = fmaxf(mx, ss[h * chunk + j]);
    mx = block_max(mx, red);
    float sum = 0.f;
    for (int j = threadIdx.x; j < cn; j += kAttnThreads) {
      const float w = expf(ss[h * chunk + j] - mx);
      ss[h * chunk + j] = w;
      sum += w;
    }
    sum = block_sum(sum, red);
    if (threadIdx.x == 0) {
      part_m[(size_t)c * Hq + g * G + h] = mx;
      part_l[(size_t)c * Hq + g * G + h] = sum;
    }
  }
  __syncthreads();

  // sum_j exp(s - m) v_j: thread t owns dimension t % D of heads t / D, t / D + slots, ...
  const int slots = kAttnThreads / D;
  const int d = threadIdx.x % D, h0 = threadIdx.x / D;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int j = 0; j < cn; ++j) {
    const float vv = load1(v + ((size_t)(j0 + j) * N + g) * D + d);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int h = h0 + i * slots;
      if (h < G) acc[i] = fmaf(ss[h * chunk + j], vv, acc[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int h = h0 + i * slots;
    if (h < G) part_acc[((size_t)c * Hq + g * G + h) * D + d] = acc[i];
  }
}

// Grid Hq, block D threads.
__global__ void attn_merge_kernel(const float* __restrict__ part_m, const float* __restrict__ part_l,
                                  const float* __restrict__ part_acc, int chunks, int Hq, int D,
                                  float* __restrict__ out) {
  const int h = blockIdx.x, d = threadIdx.x;
  float M = -FLT_MAX;
  for (int c = 0; c < chunks; ++c) M = fmaxf(M, part_m[(size_t)c * Hq + h]);
  float L = 0.f, o = 0.f;
  for (int c = 0; c < chunks; ++c) {
    const float f = expf(part_m[(size_t)c * Hq + h] - M);
    L = fmaf(part_l[(size_t)c * Hq + h], f, L);
    o = fmaf(part_acc[((size_t)c * Hq + h) * D + d], f, o);
  }
  out[(size_t)h * D + d] = o / L;
}

}  // namespace

// Tokens per chunk: at least 128, and few enough chunks for the workspace.
int attention_chunk(int n) {
  int chunk = (n + kAttnMaxChunks - 1) / kAttnMaxChunks;
  chunk = (chunk + 31) / 32 * 32;
  return chunk < 128 ? 128 : chunk;
}

cudaError_t launch_attention(rkv_ctx* c, const float* q, int n_q_heads, const void* k,
                             const void* v, int n, float* out, cudaStream_t s) {
  const Dims& d = c->d;
  const int G = n_q_heads / d.N;
  const int chunk = attention_chunk(n);
  const int chunks = (n + chunk - 1) / chunk;
  float* pm = c->attn_ws;
  float* pl = pm + (size_t)kAttnMaxChunks * n_q_heads;
  float* pa = pl + (size_t)kAttnMaxChunks * n_q_heads;
  // q [G][D] and the weights [G][chunk]: at most 8 x (128 + 1024) floats = 36 KB
  const size_t smem = sizeof(float) * ((size_t)G * d.D + (size_t)G * chunk);
  cudaEvent_t ev;
  timing_begin(c, "rkv_attention_partial_kernel", s, &ev);
  if (d.out_f32) {
    attn_partial_kernel<float><<<dim3(chunks, d.N), kAttnThreads, smem, s>>>(
        q, static_cast<const float*>(k), static_cast<const float*>(v), n, d.N, d.D, G, chunk, pm,
        pl, pa);
  } else {
    attn_partial_kernel<__nv_bfloat16><<<dim3(chunks, d.N), kAttnThreads, smem, s>>>(
        q, static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), n, d.N,
        d.D, G, chunk, pm, pl, pa);
  }
  timing_end(c, "rkv_attention_partial_kernel", s, ev);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  timing_begin(c, "rkv_attention_merge_kernel", s, &ev);
  attn_merge_kernel<<<n_q_heads, d.D, 0, s>>>(pm, pl, pa, chunks, n_q_heads, d.D, out);
  timing_end(c, "rkv_attention_merge_kernel", s, ev);
  return cudaGetLastError();
}

}  // namespace rkv
