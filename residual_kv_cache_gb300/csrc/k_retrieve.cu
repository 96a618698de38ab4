// k_retrieve.cu - global top-k L2 retrieval of references (ResidualKV notes §2.2, the
// arg top-k_i equation; k_i = min(k, |T_ref,i|), T_ref,i = references before token i).
//
// For a tile of 128 query tokens of one sequence and a tile of 256 pool slots the
// tensor cores compute the dot products a_i . r_j (bf16 operands, exact products, fp32
// accumulation in TMEM).  Two epilogue warpgroups split the 256 slots; the thread of
// each that owns query row i (one TMEM lane) turns its dot products into the ranking
// score ||r_j||^2 - 2 a_i . r_j (= ||a_i - r_j||^2 minus a per-row constant), masks
// slots whose reference is not strictly before the token, and keeps a sorted top-4;
// the second group hands its list to the first, which inserts it.  A sequence's pool
// slots hold its reference positions in increasing order, so the references before
// position p are exactly slots 0 .. ref_before[p] - 1: the mask is one compare with a
// per-row bound.  The unit's 256 squared norms are staged once in shared memory and
// read four at a time by broadcast loads.  Equal scores keep the smaller slot because
// slots are visited in increasing order with a strict comparison.  fp32 queries are
// split into three bf16 pieces (hi + mid + lo == x), so the products stay exact and the
// three partial dots accumulate into one fp32 sum.
//
// Work unit = (128-query tile, 256-slot pool tile): all units cost the same, so a
// persistent grid balances them.  Each unit leaves a sorted partial top-4 per query
// row; a merge kernel combines a row's partials in increasing slot order with the same
// strict comparison, which yields exactly the 4 smallest (distance, slot) pairs.
#include <cuda_bf16.h>
#include <float.h>

#include "tc_common.cuh"

namespace rkv {
namespace {

struct RetrieveArgs {
  const int32_t* t_seq;
  const int32_t* t_row0;
  const int32_t* t_nrt;
  const int32_t* t_u0;
  const int32_t* u_tile;
  const int32_t* u_rt;
  const int32_t* q_pos;
  const int32_t* q_dst;
  int2* part;
  int n_units;
  int nkb;      // k-blocks per piece (2d_k / 64)
  int parts;    // 1 or 3
  int R_cap, topk;
  const float* norm2;
  const int32_t* ref_before;   // [T_cap + 1] references below each position
  int32_t* ref_idx;
  int* status;
};

constexpr int kStages = 4;
// 12 warps: 0 TMA producer, 1 MMA issuer, 2 TMEM allocator, 3 idle, 4..11 epilogue in two
// groups of four; group g scans columns [128 g, 128 g + 128) of each unit's 256 slots.
constexpr int kRetrThreads = 384;
constexpr int kEpiThreads = 256;
constexpr uint32_t kBBytes = kRefTile * 128;
constexpr uint32_t kTmemCols = 2 * kRefTile;

__device__ __forceinline__ void topk_insert(float d, int j, float* bd, int* bj) {
  if (!(d < bd[3])) return;
  if (d < bd[2]) {
    bd[3] = bd[2];
    bj[3] = bj[2];
    if (d < bd[1]) {
      bd[2] = bd[1];
      bj[2] = bj[1];
      if (d < bd[0]) {
        bd[1] = bd[0];
        bj[1] = bj[0];
        bd[0] = d;
        bj[0] = j;
      } else {
        bd[1] = d;
        bj[1] = j;
      }
    } else {
      bd[2] = d;
      bj[2] = j;
    }
  } else {
    bd[3] = d;
    bj[3] = j;
  }
}

// The same insertion without branches: (d, j) goes in at the first place k where
// d < bd[k] (strict, so an equal score keeps the earlier, smaller slot), the entries from
// k on move down one, and the last falls out; nothing changes when d >= bd[3].  The four
// compares and the selects run on every lane alike, so a warp whose lanes insert at
// different places (or not at all) never splits.
__device__ __forceinline__ void topk_insert_nb(float d, int j, float* bd, int* bj) {
  const bool c0 = d < bd[0], c1 = d < bd[1], c2 = d < bd[2], c3 = d < bd[3];
  const float n3 = c2 ? bd[2] : (c3 ? d : bd[3]);
  const int m3 = c2 ? bj[2] : (c3 ? j : bj[3]);
  const float n2 = c1 ? bd[1] : (c2 ? d : bd[2]);
  const int m2 = c1 ? bj[1] : (c2 ? j : bj[2]);
  const float n1 = c0 ? bd[0] : (c1 ? d : bd[1]);
  const int m1 = c0 ? bj[0] : (c1 ? j : bj[1]);
  bd[0] = c0 ? d : bd[0];
  bj[0] = c0 ? j : bj[0];
  bd[1] = n1;
  bj[1] = m1;
  bd[2] = n2;
  bj[2] = m2;
  bd[3] = n3;
  bj[3] = m3;
}

__global__ void __launch_bounds__(kRetrThreads, 1)
    retrieve_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmP,
                    RetrieveArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kTileABytes;
  float* sN = reinterpret_cast<float*>(sB + kStages * kBBytes);   // [2][kRefTile] norms
  int4* sM = reinterpret_cast<int4*>(sN + 2 * kRefTile);          // [kTileM][2] group 1's top-4
  uint64_t* full = reinterpret_cast<uint64_t*>(sM + 2 * kTileM);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kEpiThreads / 32);         // one arrival per epilogue warp
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch(&tmQ);
    tma_prefetch(&tmP);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int kb_total = a.parts * a.nkb;

  if (warp == 0) {
    if (elect_one()) {
      Ring ring;
      int issued[kStages];
      uint32_t issued_phase[kStages];
      for (int s = 0; s < kStages; ++s) issued[s] = 0, issued_phase[s] = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < a.n_units && ok; u += gridDim.x) {
        const int t = a.u_tile[u], rt = a.u_rt[u];
        const int seq = a.t_seq[t], row0 = a.t_row0[t];
        {
          for (int kb = 0; kb < kb_total; ++kb) {
            if (!mbar_wait(&empty[ring.stage], ring.phase ^ 1u, abort_flag, a.status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[ring.stage], kTileABytes + kBBytes);
            tma_load_2d(sA + ring.stage * kTileABytes, &tmQ, &full[ring.stage], kb * kTileK, row0);
            tma_load_2d(sB + ring.stage * kBBytes, &tmP, &full[ring.stage], (kb % a.nkb) * kTileK,
                        seq * a.R_cap + rt * kRefTile);
            issued[ring.stage] = 1;
            issued_phase[ring.stage] = ring.phase;
            ring.next(kStages);
          }
        }
      }
      if (!ok)
        for (int s = 0; s < kStages; ++s)
          if (issued[s]) drain_wait(&full[s], issued_phase[s]);
    }
  } else if (warp == 1) {
    if (elect_one()) {
      constexpr uint32_t idesc = idesc_bf16_f32(kTileM, kRefTile);
      Ring ring;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, any = false;
      int last_stage = 0;
      uint32_t last_phase = 0;
      for (int u = blockIdx.x; u < a.n_units && ok; u += gridDim.x) {
        {
          if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + acc * kRefTile;
          for (int kb = 0; kb < kb_total; ++kb) {
            if (!mbar_wait(&full[ring.stage], ring.phase, abort_flag, a.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(sA + ring.stage * kTileABytes);
            const uint32_t b0 = smem_u32(sB + ring.stage * kBBytes);
#pragma unroll
            for (int k = 0; k < kTileK / 16; ++k)
              umma_bf16(d, sdesc_sw128(a0 + k * 32), sdesc_sw128(b0 + k * 32), idesc,
                        (kb | k) != 0 ? 1u : 0u);
            umma_commit(&empty[ring.stage]);
            any = true;
            last_stage = ring.stage;
            last_phase = ring.phase;
            ring.next(kStages);
          }
          if (!ok) break;
          umma_commit(&tfull[acc]);
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
      }
      if (!ok && any) drain_wait(&empty[last_stage], last_phase);
    }
  } else if (warp >= kEpiWarp0) {
    const int et = (int)threadIdx.x - kEpiWarp0 * 32;  // 0 .. kEpiThreads - 1
    const int eg = et >> 7;                            // column group
    const int row_in_tile = et & (kTileM - 1);         // TMEM lane = query row
    const uint32_t lane_base = (uint32_t)(row_in_tile & ~31) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    int k = 0;                                         // this CTA's unit count
    for (int u = blockIdx.x; u < a.n_units; u += gridDim.x, ++k) {
      const int t = a.u_tile[u], rt = a.u_rt[u];
      const int seq = a.t_seq[t], row0 = a.t_row0[t];
      const int qrow = row0 + row_in_tile;
      const int pos = a.q_pos[qrow];
      const int64_t pbase = (int64_t)seq * a.R_cap;
      // references strictly before the token: the first ref_before[pos] slots (none for
      // a padding row, pos = -1)
      const int nref = pos >= 0 ? __ldg(a.ref_before + pos) : 0;
      // the unit's squared norms into buffer k & 1; the same barrier, whose vote also
      // makes every exit uniform, orders these writes before the reads and the reads of
      // unit k - 1 (other buffer, and group 1's list) before the writes of unit k + 1
      float* nb = sN + (k & 1) * kRefTile;
      {
        const int j = rt * kRefTile + et;
        nb[et] = j < a.R_cap ? __ldg(a.norm2 + pbase + j) : 0.f;
      }
      float bd[4] = {FLT_MAX, FLT_MAX, FLT_MAX, FLT_MAX};
      int bj[4] = {-1, -1, -1, -1};
      if (!bar_red_and(1, kEpiThreads, warp_wait(&tfull[acc], acc_phase, abort_flag, a.status)))
        break;
      tc_fence_after();
      const uint32_t tacc = tmem + lane_base + (uint32_t)(acc * kRefTile);
#pragma unroll 1
      for (int c = 4 * eg; c < 4 * eg + 4; ++c) {
        const int j0 = rt * kRefTile + c * 32;
        uint32_t r[32];
        tmem_ld32(tacc + c * 32, r);
        tmem_ld_wait();
        const float4* n4 = reinterpret_cast<const float4*>(nb + c * 32);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 nv = n4[q];
          const float nn[4] = {nv.x, nv.y, nv.z, nv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = 4 * q + e;
            // slots at or after nref (references not before the token) never enter
            const float dist = j0 + i < nref ? fmaf(-2.0f, __uint_as_float(r[i]), nn[e]) : INFINITY;
            topk_insert_nb(dist, j0 + i, bd, bj);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane_id() == 0) mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
      // group 1 (the larger slots) hands its list to group 0, which inserts it in order
      // with the same strict comparison, so equal scores still keep the smaller slot
      if (eg == 1) {
        sM[2 * row_in_tile] = make_int4(__float_as_int(bd[0]), bj[0], __float_as_int(bd[1]), bj[1]);
        sM[2 * row_in_tile + 1] = make_int4(__float_as_int(bd[2]), bj[2], __float_as_int(bd[3]), bj[3]);
        bar_arrive(2, kEpiThreads);
        continue;
      }
      bar_sync(2, kEpiThreads);
      {
        const int4 e0 = sM[2 * row_in_tile], e1 = sM[2 * row_in_tile + 1];
        const float od[4] = {__int_as_float(e0.x), __int_as_float(e0.z), __int_as_float(e1.x),
                             __int_as_float(e1.z)};
        const int oj[4] = {e0.y, e0.w, e1.y, e1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (oj[i] >= 0) topk_insert(od[i], oj[i], bd, bj);
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
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One thread per retrieval-order row: merge the row's partial top-4 lists of its pool
// tiles (increasing slots) and write the final slots of real rows.
__global__ void retrieve_merge_kernel(const int2* __restrict__ part, const int32_t* __restrict__ t_nrt,
                                      const int32_t* __restrict__ t_u0,
                                      const int32_t* __restrict__ q_pos,
                                      const int32_t* __restrict__ q_dst, int m_pad, int topk,
                                      int32_t* __restrict__ ref_idx) {
  const int q = blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= m_pad || q_pos[q] < 0) return;
  const int t = q / kTileM, r = q % kTileM;
  float bd[4] = {FLT_MAX, FLT_MAX, FLT_MAX, FLT_MAX};
  int bj[4] = {-1, -1, -1, -1};
  const int u0 = t_u0[t], nrt = t_nrt[t];
  for (int k = 0; k < nrt; ++k) {
    const int4* sp = reinterpret_cast<const int4*>(part + ((int64_t)(u0 + k) * kTileM + r) * 4);
    const int4 e0 = sp[0], e1 = sp[1];
    const float d[4] = {__int_as_float(e0.x), __int_as_float(e0.z), __int_as_float(e1.x), __int_as_float(e1.z)};
    const int j[4] = {e0.y, e0.w, e1.y, e1.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (j[i] >= 0) topk_insert(d[i], j[i], bd, bj);
  }
  const int64_t dst = q_dst[q];
  for (int i = 0; i < topk; ++i) ref_idx[dst * topk + i] = bj[i];
}

}  // namespace

cudaError_t launch_retrieve_merge(rkv_ctx* c, const PassPlan& p, const int32_t* plan,
                                  cudaStream_t s) {
  if (p.m_pad == 0) return cudaSuccess;
  cudaEvent_t ev;
  timing_begin(c, "rkv_retrieve_merge_kernel", s, &ev);
  retrieve_merge_kernel<<<(p.m_pad + 127) / 128, 128, 0, s>>>(
      c->part, plan + p.off_t_nrt, plan + p.off_t_u0, plan + p.off_q_pos, plan + p.off_q_dst,
      p.m_pad, c->d.topk, c->st.ref_idx);
  cudaError_t e = cudaGetLastError();
  timing_end(c, "rkv_retrieve_merge_kernel", s, ev);
  return e;
}

cudaError_t launch_retrieve(rkv_ctx* c, const PassPlan& p, const int32_t* plan, cudaStream_t s) {
  if (p.n_units == 0) return cudaSuccess;
  const size_t smem = 1024 + (size_t)kStages * (kTileABytes + kBBytes) + 2 * kRefTile * sizeof(float) +
                      2 * kTileM * sizeof(int4) + 8 * (2 * kStages + 4) + 16;
  cudaError_t e =
      cudaFuncSetAttribute(retrieve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  RetrieveArgs a;
  a.t_seq = plan + p.off_t_seq;
  a.t_row0 = plan + p.off_t_row0;
  a.t_nrt = plan + p.off_t_nrt;
  a.t_u0 = plan + p.off_t_u0;
  a.u_tile = plan + p.off_u_tile;
  a.u_rt = plan + p.off_u_rt;
  a.q_pos = plan + p.off_q_pos;
  a.q_dst = plan + p.off_q_dst;
  a.part = c->part;
  a.n_units = p.n_units;
  a.nkb = c->d.dkv / kTileK;
  a.parts = c->d.parts;
  a.R_cap = c->d.R_cap;
  a.topk = c->d.topk;
  a.norm2 = c->st.pool_norm2;
  a.ref_before = c->ref_before_dev;
  a.ref_idx = c->st.ref_idx;
  a.status = c->status;
  const int grid = p.n_units < c->num_sms ? p.n_units : c->num_sms;
  cudaEvent_t ev;
  timing_begin(c, "rkv_retrieve_kernel", s, &ev);
  retrieve_kernel<<<grid, kRetrThreads, smem, s>>>(c->tm_q, c->tm_pool, a);
  e = cudaGetLastError();
  timing_end(c, "rkv_retrieve_kernel", s, ev);
  return e;
}

}  // namespace rkv
