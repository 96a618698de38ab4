// tc_common.cuh - pieces shared by the tcgen05 kernels: shared-memory carve-up, the
// TMA producer / MMA issuer ring protocol, and the bounded teardown.
//
// Warp roles of the encoder GEMMs (256 threads):
//   warp 0      TMA producer (one elected lane)
//   warp 1      MMA issuer (one elected lane)
//   warp 2      TMEM allocator (whole warp), idle otherwise
//   warp 3      idle
//   warps 4..7  epilogue: warp 4+w owns TMEM lanes [32w, 32w+32), i.e. tile rows.
// The retrieval (384 threads, two epilogue warpgroups) and the restore (640 threads,
// four) keep warps 0 and 1 in these roles and add epilogue warps; a warp w reads TMEM
// lanes [32 (w % 4), +32).
#pragma once
#include "ptx.cuh"
#include "rkv_internal.h"

namespace rkv {

constexpr int kThreads = 256;
constexpr int kEpiWarp0 = 4;
constexpr uint32_t kTileABytes = kTileM * 128;   // 128 rows x 64 bf16

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t s = smem_u32(p);
  return p + ((1024u - (s & 1023u)) & 1023u);
}

// Ring position (stage index and phase bit) of a multi-stage pipeline.
struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int stages) {
    if (++stage == stages) {
      stage = 0;
      phase ^= 1u;
    }
  }
};

// Warp-uniform bounded wait: lane 0 waits, the verdict is broadcast to the warp so that
// the following .sync.aligned tcgen05 instructions run with the whole warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* status) {
  int ok = 1;
  if (lane_id() == 0) ok = mbar_wait(bar, parity, abort, status) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

// After an abort, wait (bounded, ~0.1 s) until every operation that `bar` tracks with
// `parity` has landed, so no copy or MMA is left writing into a CTA that has left.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitCycles / 10) break;
  }
}

}  // namespace rkv
