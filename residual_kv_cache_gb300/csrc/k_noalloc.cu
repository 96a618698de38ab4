// k_noalloc.cu - top-k L2 retrieval of one sequence against one reference pool that
// allocates nothing: its only scratch (the per-pool-tile partial top-4 lists) lives in
// a fixed device array inside this library.
//
// Who needs it: code that must not call the CUDA allocator while it runs - a serving
// runtime that reserves all device memory up front in its own arena and may not grow
// or fragment it mid-step, or a step that must not pay cudaMalloc's implicit device
// synchronisation.  Such a caller cannot create a codec context (rkv_create allocates
// workspace), but it can still run the retrieval step on buffers it already owns.
//
// The kernel computes exactly what the compress path's retrieval computes (same
// tensor-core dot products in the same K order, same masking and tie rule), so its
// slots are identical to the ones rkv_compress stores.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <float.h>

#include <climits>
#include <mutex>

#include "tc_common.cuh"

namespace rkv {
namespace {

constexpr int kNaRefTile = 256;
constexpr int kNaStages = 4;
constexpr uint32_t kNaBBytes = kNaRefTile * 128;
// 1024 units x 128 rows x 4 (distance bits, slot) pairs of 8 bytes = 4 MiB, plus a
// 256-byte tail holding the status word used when the caller passes no flags.
constexpr int kNaMaxUnits = 1024;
constexpr size_t kNaListInts = (size_t)kNaMaxUnits * kTileM * 4 * 2;
constexpr size_t kNaScratchInts = kNaListInts + 64;

// The scratch.  Every GPU that loads the library holds these 4 MiB until the process
// exits.  Host code must not use this name as an address (it is a host-side stand-in);
// it obtains the device address with cudaGetSymbolAddress, once per device.
static __device__ __align__(256) int32_t g_noalloc_scratch[kNaScratchInts];

__device__ __forceinline__ void na_topk_insert(float d, int j, float* bd, int* bj) {
  if (!(d < bd[3])) return;
  if (d < bd[2]) {
    bd[3] = bd[2]; bj[3] = bj[2];
    if (d < bd[1]) {
      bd[2] = bd[1]; bj[2] = bj[1];
      if (d < bd[0]) {
        bd[1] = bd[0]; bj[1] = bj[0];
        bd[0] = d; bj[0] = j;
      } else {
        bd[1] = d; bj[1] = j;
      }
    } else {
      bd[2] = d; bj[2] = j;
    }
  } else {
    bd[3] = d; bj[3] = j;
  }
}

struct NaArgs {
  const int32_t* q_pos;
  int n, R, nkb, n_rt, n_units;
  const float* norm2;
  const int32_t* pool_pos;
  int2* part;          // the static scratch, as passed by the host
  int* status;
};

// Unit u = (query tile u / n_rt, pool tile u % n_rt); same roles as the compress path.
__global__ void __launch_bounds__(kThreads, 1)
    noalloc_retrieve_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmP, NaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kNaStages * kTileABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kNaStages * kNaBBytes);
  uint64_t* empty = full + kNaStages;
  uint64_t* tfull = empty + kNaStages;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  constexpr uint32_t kCols = 2 * kNaRefTile;

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kNaStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 128);
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch(&tmQ);
    tma_prefetch(&tmP);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (elect_one()) {
      Ring ring;
      int issued[kNaStages];
      uint32_t issued_phase[kNaStages];
      for (int s = 0; s < kNaStages; ++s) issued[s] = 0, issued_phase[s] = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < a.n_units && ok; u += gridDim.x) {
        const int t = u / a.n_rt, rt = u % a.n_rt;
        for (int kb = 0; kb < a.nkb; ++kb) {
          if (!mbar_wait(&empty[ring.stage], ring.phase ^ 1u, abort_flag, a.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[ring.stage], kTileABytes + kNaBBytes);
          tma_load_2d(sA + ring.stage * kTileABytes, &tmQ, &full[ring.stage], kb * kTileK, t * kTileM);
          tma_load_2d(sB + ring.stage * kNaBBytes, &tmP, &full[ring.stage], kb * kTileK, rt * kNaRefTile);
          issued[ring.stage] = 1;
          issued_phase[ring.stage] = ring.phase;
          ring.next(kNaStages);
        }
      }
      if (!ok)
        for (int s = 0; s < kNaStages; ++s)
          if (issued[s]) drain_wait(&full[s], issued_phase[s]);
    }
  } else if (warp == 1) {
    if (elect_one()) {
      constexpr uint32_t idesc = idesc_bf16_f32(kTileM, kNaRefTile);
      Ring ring;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, any = false;
      int last_stage = 0;
      uint32_t last_phase = 0;
      for (int u = blockIdx.x; u < a.n_units && ok; u += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + acc * kNaRefTile;
        for (int kb = 0; kb < a.nkb; ++kb) {
          if (!mbar_wait(&full[ring.stage], ring.phase, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + ring.stage * kTileABytes);
          const uint32_t b0 = smem_u32(sB + ring.stage * kNaBBytes);
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k)
            umma_bf16(d, sdesc_sw128(a0 + k * 32), sdesc_sw128(b0 + k * 32), idesc,
                      (kb | k) != 0 ? 1u : 0u);
          umma_commit(&empty[ring.stage]);
          any = true;
          last_stage = ring.stage;
          last_phase = ring.phase;
          ring.next(kNaStages);
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
    const int ew = warp - kEpiWarp0;
    const int row_in_tile = ew * 32 + (int)lane_id();
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < a.n_units; u += gridDim.x) {
      const int t = u / a.n_rt, rt = u % a.n_rt;
      const int q = t * kTileM + row_in_tile;
      const int pos = q < a.n ? a.q_pos[q] : -1;
      float bd[4] = {FLT_MAX, FLT_MAX, FLT_MAX, FLT_MAX};
      int bj[4] = {-1, -1, -1, -1};
      if (!warp_wait(&tfull[acc], acc_phase, abort_flag, a.status)) break;
      tc_fence_after();
      const uint32_t tacc = tmem + ((uint32_t)(ew * 32) << 16) + (uint32_t)(acc * kNaRefTile);
#pragma unroll 1
      for (int c = 0; c < kNaRefTile / 32; ++c) {
        const int j0 = rt * kNaRefTile + c * 32;
        const int jl = j0 + (int)lane_id();
        int32_t pl = INT_MAX;
        float nl = 0.f;
        if (jl < a.R) {
          pl = __ldg(a.pool_pos + jl);
          nl = __ldg(a.norm2 + jl);
        }
        uint32_t r[32];
        tmem_ld32(tacc + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int32_t pj = __shfl_sync(0xffffffffu, pl, i);
          const float nj = __shfl_sync(0xffffffffu, nl, i);
          const float dist = fmaf(-2.0f, __uint_as_float(r[i]), nj);
          if (pj < pos) na_topk_insert(dist, j0 + i, bd, bj);
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
      int4* dp = reinterpret_cast<int4*>(a.part + ((int64_t)u * kTileM + row_in_tile) * 4);
      dp[0] = make_int4(__float_as_int(bd[0]), bj[0], __float_as_int(bd[1]), bj[1]);
      dp[1] = make_int4(__float_as_int(bd[2]), bj[2], __float_as_int(bd[3]), bj[3]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// One thread per query: merge its pool tiles' partial lists (increasing slots) and
// write the final slots.  Every partial it reads was written earlier in this call.  If a
// wait of the retrieval kernel gave up (RKV_FLAG_TIMEOUT in the call's status word), some
// partial lists may be stale, so every slot of the output is written as -1 instead.
__global__ void noalloc_merge_kernel(const int2* __restrict__ part, const int32_t* __restrict__ q_pos,
                                     int n, int n_rt, int topk, const int* status,
                                     int32_t* __restrict__ out_idx) {
  const int q = blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= n) return;
  if (*reinterpret_cast<const volatile int*>(status) & RKV_FLAG_TIMEOUT) {
    for (int i = 0; i < topk; ++i) out_idx[(int64_t)q * topk + i] = -1;
    return;
  }
  const int t = q / kTileM, r = q % kTileM;
  float bd[4] = {FLT_MAX, FLT_MAX, FLT_MAX, FLT_MAX};
  int bj[4] = {-1, -1, -1, -1};
  for (int k = 0; k < n_rt; ++k) {
    const int4* sp = reinterpret_cast<const int4*>(part + ((int64_t)(t * n_rt + k) * kTileM + r) * 4);
    const int4 e0 = sp[0], e1 = sp[1];
    const float d[4] = {__int_as_float(e0.x), __int_as_float(e0.z), __int_as_float(e1.x), __int_as_float(e1.z)};
    const int j[4] = {e0.y, e0.w, e1.y, e1.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (j[i] >= 0) na_topk_insert(d[i], j[i], bd, bj);
  }
  for (int i = 0; i < topk; ++i) out_idx[(int64_t)q * topk + i] = bj[i];
}

// ---- per-device set-up: the device address of the scratch, and a status word inside it
struct DeviceSlot {
  std::mutex mu;
  void* scratch = nullptr;   // set once the look-up has succeeded
};
constexpr int kMaxDevices = 64;
DeviceSlot g_slots[kMaxDevices];

// The status word used when the caller passes no flags: the scratch's tail.
constexpr size_t kStatusOffsetInts = kNaListInts;

PFN_cuTensorMapEncodeTiled_v12000 na_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool na_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const void* base, uint64_t inner,
            uint64_t rows, uint32_t box_rows) {
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64u, box_rows};
  cuuint32_t es[2] = {1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

rkv_status noalloc_retrieve(const void* queries, const int32_t* q_pos, int32_t n, const void* pool,
                            const float* pool_norm2, const int32_t* pool_pos, int32_t R, int32_t d,
                            int32_t topk, int32_t* out_idx, int32_t* flags, cudaStream_t s,
                            const char** why) {
  if (n < 0 || R < 0) return *why = "n and R must be >= 0", RKV_EINVAL;
  if (n == 0) return RKV_OK;
  if (!queries || !q_pos || !pool || !pool_norm2 || !pool_pos || !out_idx)
    return *why = "NULL pointer", RKV_EINVAL;
  if (R == 0) return *why = "empty reference pool", RKV_EEMPTYPOOL;
  if (d <= 0 || d % 64 != 0) return *why = "d must be a positive multiple of 64", RKV_EINVAL;
  if (topk < 1 || topk > 4) return *why = "topk must be in 1..4", RKV_EINVAL;
  if ((reinterpret_cast<uintptr_t>(queries) | reinterpret_cast<uintptr_t>(pool)) & 15u)
    return *why = "queries and pool must be 16-byte aligned", RKV_EALIGN;
  const int n_rt = (R + kNaRefTile - 1) / kNaRefTile;
  const int64_t units = (int64_t)((n + kTileM - 1) / kTileM) * n_rt;
  if (units > kNaMaxUnits)
    return *why = "ceil(n/128) * ceil(R/256) exceeds the 1024 tiles of the fixed scratch "
                  "(for example n <= 2048 queries with R <= 16384 references)",
           RKV_ECAPACITY;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return *why = "no usable current device", RKV_ECUDA;
  DeviceSlot& slot = g_slots[dev];
  void* scratch = nullptr;
  {
    // With this device current: the device address of the scratch array.  Only a
    // successful look-up is kept, so a call that failed (for instance one made during a
    // stream capture) leaves the next call free to try again.
    std::lock_guard<std::mutex> lock(slot.mu);
    if (slot.scratch == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return *why = "cudaGetSymbolAddress of the scratch failed", RKV_ECUDA;
      }
      slot.scratch = p;
    }
    scratch = slot.scratch;
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc = na_encoder();
  if (!enc) return *why = "cuTensorMapEncodeTiled is unavailable", RKV_ECUDA;
  CUtensorMap tmQ, tmP;
  if (!na_map(enc, &tmQ, queries, d, n, kTileM) || !na_map(enc, &tmP, pool, d, R, kNaRefTile))
    return *why = "cuTensorMapEncodeTiled rejected the operands", RKV_ECUDA;

  NaArgs a;
  a.q_pos = q_pos;
  a.n = n;
  a.R = R;
  a.nkb = d / kTileK;
  a.n_rt = n_rt;
  a.n_units = (int)units;
  a.norm2 = pool_norm2;
  a.pool_pos = pool_pos;
  a.part = static_cast<int2*>(scratch);
  a.status = flags ? flags : static_cast<int*>(scratch) + kStatusOffsetInts;
  const size_t smem = 1024 + (size_t)kNaStages * (kTileABytes + kNaBBytes) + 8 * (2 * kNaStages + 4) + 16;
  if (cudaFuncSetAttribute(noalloc_retrieve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return *why = "cudaFuncSetAttribute failed", RKV_ECUDA;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return *why = "cudaDeviceGetAttribute failed", RKV_ECUDA;
  const int grid = units < sms ? (int)units : sms;
  // without caller flags, the call's status word is the scratch's own: cleared here so
  // that it holds this call's verdict alone
  if (!flags && cudaMemsetAsync(a.status, 0, sizeof(int), s) != cudaSuccess)
    return *why = "clearing the status word failed", RKV_ECUDA;
  noalloc_retrieve_kernel<<<grid, kThreads, smem, s>>>(tmQ, tmP, a);
  if (cudaGetLastError() != cudaSuccess) return *why = "retrieval launch failed", RKV_ECUDA;
  noalloc_merge_kernel<<<(n + 127) / 128, 128, 0, s>>>(a.part, q_pos, n, n_rt, topk, a.status,
                                                        out_idx);
  if (cudaGetLastError() != cudaSuccess) return *why = "merge launch failed", RKV_ECUDA;
  return RKV_OK;
}

}  // namespace rkv

extern "C" rkv_status rkv_retrieve_noalloc(const void* queries, const int32_t* q_pos, int32_t n,
                                           const void* pool, const float* pool_norm2,
                                           const int32_t* pool_pos, int32_t R, int32_t d,
                                           int32_t topk, int32_t* out_idx, int32_t* flags,
                                           void* stream) {
  const char* why = "";
  const rkv_status st = rkv::noalloc_retrieve(queries, q_pos, n, pool, pool_norm2, pool_pos, R, d,
                                              topk, out_idx, flags,
                                              static_cast<cudaStream_t>(stream), &why);
  if (st != RKV_OK) rkv::set_error(why);
  return st;
}
