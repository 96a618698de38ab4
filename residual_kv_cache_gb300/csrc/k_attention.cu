// k_attention.cu - sparse-layer attention over restored K/V (ResidualKV notes §2.7, the
// output equation o = softmax(q K_hat^T / sqrt(D)) V_hat over the selected tokens).
//
// Decode attention is a few dot products per token against K/V rows that a restore has
// just written (they are still in L2), so the work is split over the tokens, not over
// the heads: a CTA takes one chunk of selected tokens and one key/value head, scores
// the chunk against every query head of that head's group, and keeps a chunk-local
// softmax (its maximum m, its sum l of exp(s - m), and sum exp(s - m) v).  The last CTA
// of each key/value head to finish (a counter after a fence) merges that head's chunks:
// M = max m_c, L = sum l_c e^(m_c - M), o = sum acc_c e^(m_c - M) / L, and puts the
// counter back to zero for the next call.  Everything is fp32; exp is the library expf.
#include <cuda_bf16.h>
#include <stdint.h>

#include <cfloat>

#include <cooperative_groups.h>

#include "ptx.cuh"
#include "rkv_internal.h"

namespace rkv {
namespace cg = cooperative_groups;
namespace {

constexpr int kAttnThreads = 256;
constexpr int kWarps = kAttnThreads / 32;
constexpr int kAttnCtasPerSm = 3;             // resident CTAs per SM (registers <= 85)

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  v = red[0];
  for (int i = 1; i < kWarps; ++i) v = fmaxf(v, red[i]);
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
  for (int i = 0; i < kWarps; ++i) v += red[i];
  return v;
}

// Eight consecutive elements as floats (16-byte or 32-byte aligned).
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

// Four consecutive elements (D = 128: one lane's share of a row) or two (D = 64).
__device__ __forceinline__ void load_lane(const __nv_bfloat16* p, int n, float* f) {
  if (n == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    f[0] = __uint_as_float(u.x << 16), f[1] = __uint_as_float(u.x & 0xFFFF0000u);
    f[2] = __uint_as_float(u.y << 16), f[3] = __uint_as_float(u.y & 0xFFFF0000u);
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    f[0] = __uint_as_float(u << 16), f[1] = __uint_as_float(u & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void load_lane(const float* p, int n, float* f) {
  if (n == 4) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w;
  } else {
    const float2 a = *reinterpret_cast<const float2*>(p);
    f[0] = a.x, f[1] = a.y;
  }
}

}  // namespace

// Shared memory of one CTA, in floats: q [G][4][D/4 + 4] (quarters padded apart),
// the weights [G][chunk] and the warp sums [8][G][D].
static size_t attention_smem_floats(int G, int D, int chunk) {
  return (size_t)G * (D + 16) + (size_t)G * chunk + (size_t)kWarps * G * D;
}

namespace {

// Grid (chunks, N).  part_m, part_l: [chunks][Hq]; part_acc: [chunks][Hq][D];
// count [N]: finished chunks of each key/value head (zero between calls).
template <typename T, int D>
__global__ void __launch_bounds__(kAttnThreads, kAttnCtasPerSm)
    attn_kernel(const float* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                int n, int N, int G, int chunk, float* __restrict__ part_m,
                float* __restrict__ part_l, float* __restrict__ part_acc, int* __restrict__ count,
                float* __restrict__ out) {
  extern __shared__ float sm[];
  __shared__ float red[kWarps];
  __shared__ int is_last;
  __shared__ float Ls[kAttnMaxGroup];
  constexpr int dq = D / 4;                   // dimensions per quarter row
  constexpr int qstride = dq + 4;             // padded so the four quarters hit distinct banks
  float* qs = sm;                             // [G][4][qstride]
  float* ss = sm + G * 4 * qstride;           // [G][chunk]
  float* wsum = ss + G * chunk;               // [8][G][D]
  const int c = blockIdx.x, g = blockIdx.y;
  const int Hq = G * N;
  const int j0 = c * chunk;
  const int cn = min(chunk, n - j0);
  const float scale = rsqrtf((float)D);
  for (int i = threadIdx.x; i < G * D; i += kAttnThreads) {
    const int h = i / D, d = i % D;
    qs[(h * 4 + d / dq) * qstride + d % dq] = q[(size_t)(g * G + h) * D + d] * scale;
  }
  __syncthreads();

  // scores: four threads per token, each a quarter of the row, so that a warp
  // instruction reads contiguous quarter rows of eight tokens
  {
    const int quarter = threadIdx.x & 3;
    const float* qq = qs + quarter * qstride;
    const int cn_pad = (cn + kAttnThreads / 4 - 1) / (kAttnThreads / 4) * (kAttnThreads / 4);
    for (int j = threadIdx.x >> 2; j < cn_pad; j += kAttnThreads / 4) {
      float s[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) s[h] = 0.f;
      if (j < cn) {
        const T* kr = k + ((size_t)(j0 + j) * N + g) * D + quarter * dq;
#pragma unroll
        for (int d = 0; d < dq; d += 8) {
          float kf[8];
          load8(kr + d, kf);
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            if (h < G) {
#pragma unroll
              for (int e = 0; e < 8; ++e) s[h] = fmaf(qq[h * 4 * qstride + d + e], kf[e], s[h]);
            }
          }
        }
      }
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        if (h < G) {
          s[h] += __shfl_xor_sync(0xffffffffu, s[h], 1);
          s[h] += __shfl_xor_sync(0xffffffffu, s[h], 2);
          if (j < cn && quarter == 0) ss[h * chunk + j] = s[h];
        }
      }
    }
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

  // sum_j exp(s - m) v_j: warp w takes tokens w, w + 8, ...; lane l the dimensions
  // [l * D / 32, (l + 1) * D / 32), so that a warp reads a whole V row per token
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int dpl = D / 32;                      // 4 or 2 dimensions per lane
  float acc[8][4];
#pragma unroll
  for (int h = 0; h < 8; ++h)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[h][e] = 0.f;
#pragma unroll 8
  for (int j = warp; j < cn; j += kWarps) {
    float vf[4] = {0.f, 0.f, 0.f, 0.f};
    load_lane(v + ((size_t)(j0 + j) * N + g) * D + lane * dpl, dpl, vf);
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      if (h < G) {
        const float w = ss[h * chunk + j];
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[h][e] = fmaf(w, vf[e], acc[h][e]);
      }
    }
  }
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    if (h < G) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (e < dpl) wsum[(warp * G + h) * D + lane * dpl + e] = acc[h][e];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += kAttnThreads) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t += wsum[w * G * D + i];
    part_acc[((size_t)c * Hq + g * G) * D + i] = t;
  }

  // the last CTA of this key/value head merges its chunks
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(&count[g], 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  const int C = gridDim.x;
  // every chunk's (m, l) of the group's heads in one pass, into the warp-sum area
  // ([2][G][kAttnMaxChunks] <= 8 G D floats); then M_h, the factors e^(m_c - M_h) in
  // place of m, and L_h into Ls
  float* fac = wsum;                               // [G][kAttnMaxChunks]: m, then factors
  float* lc = wsum + G * kAttnMaxChunks;           // [G][kAttnMaxChunks]: l
  for (int i = threadIdx.x; i < G * C; i += kAttnThreads) {
    const int h = i / C, cc = i % C;
    fac[h * kAttnMaxChunks + cc] = __ldcg(part_m + (size_t)cc * Hq + g * G + h);
    lc[h * kAttnMaxChunks + cc] = __ldcg(part_l + (size_t)cc * Hq + g * G + h);
  }
  __syncthreads();
  // warp h (< G <= 8) reduces head h
  if (warp < G) {
    float mx = -FLT_MAX;
    for (int cc = lane; cc < C; cc += 32) mx = fmaxf(mx, fac[warp * kAttnMaxChunks + cc]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float L = 0.f;
    for (int cc = lane; cc < C; cc += 32) {
      const float f = expf(fac[warp * kAttnMaxChunks + cc] - mx);
      fac[warp * kAttnMaxChunks + cc] = f;
      L = fmaf(lc[warp * kAttnMaxChunks + cc], f, L);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) Ls[warp] = L;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += kAttnThreads) {
    const int h = i / D;
    const float* pa = part_acc + (size_t)(g * G) * D + i;
    float o = 0.f;
#pragma unroll 16
    for (int cc = 0; cc < C; ++cc)
      o = fmaf(__ldcg(pa + (size_t)cc * Hq * D), fac[h * kAttnMaxChunks + cc], o);
    out[(size_t)(g * G) * D + i] = o / Ls[h];
  }
  if (threadIdx.x == 0) count[g] = 0;                // ready for the next call
}

// Merge of the fused restore + attention's partials (one per 128-token tile and query
// head; maxima in base-2 units).  A cluster of kMergeSlices CTAs produces dimensions
// [32 c, 32 c + 32) of query head h.  Warp w of CTA s takes tiles s + S (w + 8 j) in one
// pass, keeping a running (M, L, o) (lane = dimension): per tile, M' = max(M, m_t), then
// L = L 2^(M - M') + l_t 2^(m_t - M') and o likewise, so every load is independent of the
// others.  The eight warps' triples are combined the same way in shared memory, and CTA 0
// combines the slices' triples from the other CTAs' shared memory.
constexpr int kMergeSlices = 8;
constexpr int kMergeThreads = 256;
constexpr int kMergeMaxTiles = kAttnMaxTokens / kTileM;

struct Triple {
  float M, L, o;
};

__device__ __forceinline__ void merge_into(Triple& a, float m, float l, float o) {
  const float M = fmaxf(a.M, m);
  const float fa = ex2_approx(a.M - M), fb = ex2_approx(m - M);   // 0 for -FLT_MAX terms
  a.L = fmaf(a.L, fa, l * fb);
  a.o = fmaf(a.o, fa, o * fb);
  a.M = M;
}

__global__ void __launch_bounds__(kMergeThreads)
    attend_merge_kernel(const float* __restrict__ pm, const float* __restrict__ pl,
                        const float* __restrict__ po, int tiles, int Hq, float* __restrict__ out) {
  __shared__ float wm[8], wl[8], wo[8][32];
  __shared__ float slice[34];                      // M_s, L_s, o_s[32]
  cg::cluster_group cluster = cg::this_cluster();
  pdl_launch_dependents();
  pdl_wait_previous_grid();                        // the partials of the fused launch
  const int s = blockIdx.x, c = blockIdx.y, h = blockIdx.z;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  Triple acc{-FLT_MAX, 0.f, 0.f};
#pragma unroll 4
  for (int t = s + kMergeSlices * w; t < tiles; t += kMergeSlices * 8) {
    const size_t i = (size_t)t * Hq + h;
    merge_into(acc, __ldcg(pm + i), __ldcg(pl + i), __ldcg(po + i * 128 + c * 32 + l));
  }
  if (l == 0) wm[w] = acc.M, wl[w] = acc.L;
  wo[w][l] = acc.o;
  __syncthreads();
  if (w == 0) {
    Triple t{-FLT_MAX, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 8; ++i) merge_into(t, wm[i], wl[i], wo[i][l]);
    slice[2 + l] = t.o;
    if (l == 0) slice[0] = t.M, slice[1] = t.L;
  }
  cluster.sync();                                  // every slice is in its CTA's memory
  if (s == 0 && w == 0) {
    Triple t{-FLT_MAX, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < kMergeSlices; ++r) {
      const float* sr = cluster.map_shared_rank(slice, r);
      merge_into(t, sr[0], sr[1], sr[2 + l]);
    }
    out[(size_t)h * 128 + c * 32 + l] = t.o / t.L;
  }
  cluster.sync();                                  // CTA 0 has read every slice
}

}  // namespace

cudaError_t launch_attend_merge(rkv_ctx* c, const float* pm, const float* pl, const float* po,
                                int tiles, int n_q_heads, float* out, cudaStream_t s) {
  if (tiles < 1 || tiles > kMergeMaxTiles) return cudaErrorInvalidValue;
  cudaEvent_t ev;
  timing_begin(c, "rkv_attend_merge_kernel", s, &ev);
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(kMergeSlices, 4, n_q_heads);
  lc.blockDim = dim3(kMergeThreads);
  lc.dynamicSmemBytes = 0;
  lc.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kMergeSlices;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&lc, attend_merge_kernel, pm, pl, po, tiles, n_q_heads, out);
  if (e == cudaSuccess) e = cudaGetLastError();
  timing_end(c, "rkv_attend_merge_kernel", s, ev);
  return e;
}

// Tokens per chunk: enough chunks for one resident wave of CTAs over the N key/value
// heads (kAttnCtasPerSm per SM), at most 1024 tokens (the weights' shared memory) and
// at most kAttnMaxChunks chunks (the workspace).
int attention_chunk(int n, int N, int num_sms) {
  int target = kAttnCtasPerSm * num_sms / N;
  target = target < 1 ? 1 : (target > kAttnMaxChunks ? kAttnMaxChunks : target);
  int chunk = (n + target - 1) / target;
  chunk = (chunk + 31) / 32 * 32;
  if (chunk > 1024) chunk = 1024;
  const int floor_chunk = (n + kAttnMaxChunks - 1) / kAttnMaxChunks;
  return chunk < floor_chunk ? (floor_chunk + 31) / 32 * 32 : chunk;
}

template <typename T, int D>
cudaError_t launch_attn(const float* q, const void* k, const void* v, int n, int N, int G,
                        int chunk, int chunks, float* pm, float* pl, float* pa, int* count,
                        float* out, size_t smem, int maxb, cudaStream_t s) {
  // the shared-memory opt-in is a per-device function attribute: set it once per device
  static unsigned set_on = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 32 && !((set_on >> dev) & 1u)) {
    e = cudaFuncSetAttribute(attn_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, maxb);
    if (e != cudaSuccess) return e;
    set_on |= 1u << dev;
  }
  attn_kernel<T, D><<<dim3(chunks, N), kAttnThreads, smem, s>>>(
      q, static_cast<const T*>(k), static_cast<const T*>(v), n, N, G, chunk, pm, pl, pa, count,
      out);
  return cudaGetLastError();
}

cudaError_t launch_attention(rkv_ctx* c, const float* q, int n_q_heads, const void* k,
                             const void* v, int n, float* out, cudaStream_t s) {
  const Dims& d = c->d;
  const int G = n_q_heads / d.N;
  const int chunk = attention_chunk(n, d.N, c->num_sms);
  const int chunks = (n + chunk - 1) / chunk;
  float* pm = c->attn_ws;
  float* pl = pm + (size_t)kAttnMaxChunks * n_q_heads;
  float* pa = pl + (size_t)kAttnMaxChunks * n_q_heads;
  // at most 8 x (144 + 1024 + 8 x 128) floats = 68.5 KB
  const size_t smem = sizeof(float) * attention_smem_floats(G, d.D, chunk);
  const int maxb = (int)(sizeof(float) * attention_smem_floats(kAttnMaxGroup, 128, 1024));
  cudaEvent_t ev;
  timing_begin(c, "rkv_attention_kernel", s, &ev);
  cudaError_t e;
  if (d.out_f32)
    e = d.D == 128 ? launch_attn<float, 128>(q, k, v, n, d.N, G, chunk, chunks, pm, pl, pa,
                                             c->attn_count, out, smem, maxb, s)
                   : launch_attn<float, 64>(q, k, v, n, d.N, G, chunk, chunks, pm, pl, pa,
                                            c->attn_count, out, smem, maxb, s);
  else
    e = d.D == 128 ? launch_attn<__nv_bfloat16, 128>(q, k, v, n, d.N, G, chunk, chunks, pm, pl,
                                                     pa, c->attn_count, out, smem, maxb, s)
                   : launch_attn<__nv_bfloat16, 64>(q, k, v, n, d.N, G, chunk, chunks, pm, pl,
                                                    pa, c->attn_count, out, smem, maxb, s);
  timing_end(c, "rkv_attention_kernel", s, ev);
  return e;
}

}  // namespace rkv
