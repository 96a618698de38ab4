// rkv_api.cu - host side of the C ABI declared in include/rkv.h: validation, planning
// of compress passes, storage initialisation, tensor maps, RoPE tables, launches and
// instrumentation.  No method arithmetic happens here except the float64 RoPE tables.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "rkv_internal.h"

using namespace rkv;

namespace {

thread_local std::string g_err;

rkv_status fail(rkv_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

#define CUDA_OK(call)                                                                    \
  do {                                                                                  \
    cudaError_t e_ = (call);                                                            \
    if (e_ != cudaSuccess)                                                              \
      return fail(RKV_ECUDA, "%s failed: %s", #call, cudaGetErrorString(e_));          \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool get_encoder() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// 2-D bf16 tensor map with the 128-byte swizzle, box = {64 elements, box_rows}.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
              uint64_t row_stride_bytes, uint32_t box_rows) {
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {64u, box_rows};
  cuuint32_t es[2] = {1u, 1u};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Calls fn(p) for every reference position p < T, in increasing order, and returns
// their number (ResidualKV notes §2.6): the sink tokens 0 .. sink-1, then p_0 = sink,
// p_{m+1} = p_m + s0 + floor(alpha * (p_m - sink)), the product taken in binary64.
template <class F>
int64_t walk_schedule(int T, int s0, double alpha, int sink, F fn) {
  int64_t n = 0;
  for (int p = 0; p < sink && p < T; ++p, ++n) fn(p);
  for (int64_t p = sink; p < T; ++n) {
    fn((int)p);
    p = p + s0 + (int64_t)std::floor(alpha * (double)(p - sink));
  }
  return n;
}

rkv_status derive(const rkv_config* c, Dims* d) {
  if (!c) return fail(RKV_EINVAL, "config is NULL");
  d->N = c->n_kv_heads;
  d->D = c->head_dim;
  d->dk = c->n_kv_heads * c->head_dim;
  d->dkv = 2 * d->dk;
  d->dc = c->d_c;
  d->dff = c->d_ff;
  d->topk = c->topk;
  d->group = c->group;
  d->bits = c->bits;
  d->stride = c->ref_stride;
  d->B = c->batch;
  d->T_cap = c->max_tokens;
  d->R_cap = c->max_refs;
  d->kv_f32 = c->kv_dtype == RKV_F32;
  d->out_f32 = c->out_dtype == RKV_F32;
  d->parts = d->kv_f32 ? 3 : 1;
  if (d->N <= 0 || !(d->D == 64 || d->D == 128))
    return fail(RKV_EINVAL, "head_dim must be 64 or 128 and n_kv_heads > 0");
  if (d->dkv % 256 != 0) return fail(RKV_EINVAL, "2*N*D must be a multiple of 256");
  if (d->dc <= 0 || d->dc % 64 != 0 || d->dc > 512)
    return fail(RKV_EINVAL, "d_c must be a positive multiple of 64, at most 512");
  if (d->dff <= 0 || d->dff % 128 != 0) return fail(RKV_EINVAL, "d_ff must be a positive multiple of 128");
  if (d->topk < 1 || d->topk > 4) return fail(RKV_EINVAL, "topk must be in 1..4");
  if (d->group != 32) return fail(RKV_EINVAL, "group must be 32");
  if (!(d->bits == 4 || d->bits == 2 || d->bits == 16)) return fail(RKV_EINVAL, "bits must be 4, 2 or 16");
  if (d->stride < 1) return fail(RKV_EINVAL, "ref_stride must be >= 1");
  if (!(c->ref_alpha >= 0.0 && c->ref_alpha <= 1e6))
    return fail(RKV_EINVAL, "ref_alpha must be in [0, 1e6]");
  if (c->ref_sink < 0) return fail(RKV_EINVAL, "ref_sink must be >= 0");
  if (!(c->mean_precompute == 0 || c->mean_precompute == 1))
    return fail(RKV_EINVAL, "mean_precompute must be 0 or 1");
  d->mean_pre = c->mean_precompute;
  d->alpha = c->ref_alpha;
  d->sink = c->ref_sink;
  d->fixed = c->ref_alpha == 0.0 && c->ref_sink == 0;
  if (!(c->kv_dtype == RKV_F32 || c->kv_dtype == RKV_BF16) ||
      !(c->out_dtype == RKV_F32 || c->out_dtype == RKV_BF16))
    return fail(RKV_EINVAL, "kv_dtype / out_dtype must be RKV_F32 or RKV_BF16");
  if (!(c->rope_base > 1.0)) return fail(RKV_EINVAL, "rope_base must be > 1");
  if (d->B < 1 || d->T_cap < 1 || d->R_cap < 0)
    return fail(RKV_EINVAL, "batch and max_tokens must be >= 1, max_refs >= 0");
  d->n_sched = (int)walk_schedule(d->T_cap, d->stride, d->alpha, d->sink, [](int) {});
  if (d->R_cap == 0) d->R_cap = d->n_sched;
  if (d->R_cap < d->n_sched)
    return fail(RKV_EINVAL, "max_refs %d is below the %d reference positions under max_tokens",
                d->R_cap, d->n_sched);
  if ((int64_t)d->B * d->T_cap > INT32_MAX || (int64_t)d->B * d->R_cap > INT32_MAX)
    return fail(RKV_EINVAL, "batch * max_tokens too large");
  d->G = d->dc / d->group;
  d->code_bytes = d->bits == 16 ? 2 * d->dc : d->dc * d->bits / 8;
  d->n_hi = (d->T_cap + kRopeLo - 1) / kRopeLo;
  return RKV_OK;
}

// ------------------------------------------------------------------ staging
// Double-buffered pinned staging: before rewriting buffer b, wait for the copy that
// last read it (normally long finished).
int32_t* staging_acquire(rkv_ctx* c, int* which) {
  const int b = c->plan_flip;
  c->plan_flip ^= 1;
  cudaEventSynchronize(c->plan_copied[b]);
  *which = b;
  return c->plan_host[b];
}

// The device pulls a staged plan straight from the mapped pinned buffer with loads, so
// that the upload never queues behind a large host-to-device transfer that the caller
// runs on the copy engines at the same time (a copy-engine memcpy would).
__global__ void stage_pull_kernel(const int32_t* __restrict__ src, int32_t* __restrict__ dst, int n) {
  const int stride = gridDim.x * blockDim.x;
  const int n4 = n >> 2;
  const int4* s4 = reinterpret_cast<const int4*>(src);
  int4* d4 = reinterpret_cast<int4*>(dst);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) d4[i] = s4[i];
  for (int i = 4 * n4 + blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) dst[i] = src[i];
}

// Upload ints [first, first + n_ints) of staging buffer b; the buffer is free again once
// the event recorded after its last upload has completed.
cudaError_t staging_upload(rkv_ctx* c, int b, int first, int n_ints, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  if (n_ints <= 0) return cudaEventRecord(c->plan_copied[b], s);
  if (c->plan_host_dev[b] != nullptr && (first & 3) == 0) {
    // 16-byte aligned start (both buffers are): 256 threads per block, enough blocks
    // for the size (at most one wave)
    int blocks = (n_ints / 4 + 255) / 256;
    if (blocks < 1) blocks = 1;
    if (blocks > c->num_sms) blocks = c->num_sms;
    cudaEvent_t ev;
    timing_begin(c, "rkv_stage_pull_kernel", s, &ev);
    stage_pull_kernel<<<blocks, 256, 0, s>>>(c->plan_host_dev[b] + first, c->plan_dev[b] + first, n_ints);
    e = cudaGetLastError();
    timing_end(c, "rkv_stage_pull_kernel", s, ev);
  } else {
    e = cudaMemcpyAsync(c->plan_dev[b] + first, c->plan_host[b] + first, sizeof(int32_t) * n_ints,
                        cudaMemcpyHostToDevice, s);
  }
  if (e != cudaSuccess) return e;
  return cudaEventRecord(c->plan_copied[b], s);
}


}  // namespace

namespace rkv {

void set_error(const char* msg) { g_err = msg ? msg : ""; }

void timing_begin(rkv_ctx* c, const char* name, cudaStream_t s, cudaEvent_t* start) {
  c->launches++;
  *start = nullptr;
  if (!c->timing) return;
  if (cudaEventCreate(start) != cudaSuccess) {
    *start = nullptr;
    return;
  }
  cudaEventRecord(*start, s);
}

void timing_end(rkv_ctx* c, const char* name, cudaStream_t s, cudaEvent_t start) {
  if (!c->timing || !start) return;
  cudaEvent_t stop;
  if (cudaEventCreate(&stop) != cudaSuccess) return;
  cudaEventRecord(stop, s);
  TimingSlot* slot = nullptr;
  for (auto& t : c->timings)
    if (t.name == name) slot = &t;
  if (!slot) {
    c->timings.emplace_back();
    slot = &c->timings.back();
    slot->name = name;
  }
  slot->launches++;
  slot->pending.push_back(start);
  slot->pending.push_back(stop);
}

}  // namespace rkv

namespace {

// One pass over the rows of an rkv_compress call (branch-free, so that it vectorises):
// the checks that need no per-sequence state, and the shape of the sequence ids.
struct RowScan {
  bool bad;       // a row breaks a per-row precondition
  bool grouped;   // the sequence ids never decrease
  int runs;       // runs of equal sequence ids
  int max_pos;    // largest position (meaningful when runs == 1)
};

// kSchedule: 0 fixed power-of-two stride, 1 fixed stride, 2 any schedule (ref_before).
template <int kSchedule>
RowScan scan_compress_rows(const rkv::Dims& d, const int32_t* ref_before, const int32_t* src_rows,
                           const int32_t* seq, const int32_t* pos, int n) {
  const unsigned smask = (unsigned)d.stride - 1u;
  unsigned bad = 0, dec = 0;
  int changes = 0, max_pos = 0;
  for (int i = 0; i < n; ++i) {
    const int s = seq[i], p = pos[i];
    const unsigned p_bad = (unsigned)p >= (unsigned)d.T_cap;
    unsigned is_ref;
    if (kSchedule == 0) {
      is_ref = ((unsigned)p & smask) == 0;
    } else if (kSchedule == 1) {
      is_ref = p % d.stride == 0;
    } else {
      const int pc = p_bad ? 0 : p;
      is_ref = ref_before[pc + 1] != ref_before[pc];
    }
    bad |= (unsigned)((unsigned)s >= (unsigned)d.B) | p_bad | is_ref;
    max_pos = p > max_pos ? p : max_pos;
  }
  for (int i = 1; i < n; ++i) {
    dec |= (unsigned)(seq[i] < seq[i - 1]);
    changes += seq[i] != seq[i - 1];
  }
  if (src_rows)
    for (int i = 0; i < n; ++i) bad |= (unsigned)src_rows[i] >> 31;
  return {bad != 0, dec == 0, changes + 1, max_pos};
}

// Whether the rows of a pool append are one sequence's next n reference slots in order
// (in range, reference positions, non-negative sources); branch-free over the rows.
bool append_rows_ok_one_seq(const rkv_ctx* c, const int32_t* src_rows, const int32_t* seq,
                            const int32_t* pos, int n) {
  const rkv::Dims& d = c->d;
  const int s = seq[0];
  if ((unsigned)s >= (unsigned)d.B) return false;
  const int base = c->pool_count[s];
  if ((int64_t)base + n > d.R_cap) return false;
  const int32_t* __restrict__ rb = c->ref_before.data();
  unsigned bad = 0;
  for (int i = 0; i < n; ++i) {
    const int p = pos[i];
    const unsigned p_bad = (unsigned)p >= (unsigned)d.T_cap;
    const int pc = p_bad ? 0 : p;
    const int slot = rb[pc];
    bad |= (unsigned)(seq[i] != s) | p_bad | (unsigned)(rb[pc + 1] == slot) |
           (unsigned)(slot != base + i);
  }
  if (src_rows)
    for (int i = 0; i < n; ++i) bad |= (unsigned)src_rows[i] >> 31;
  return bad == 0;
}

// Whether some row's sequence has no reference, or lacks references before the row's
// position (the references before p are the ceil(p / stride) positions 0, stride, ...).
bool compress_pools_bad(const rkv_ctx* c, const RowScan& r, const int32_t* seq,
                        const int32_t* pos, int n) {
  // ref_before is non-decreasing, so one sequence needs only its largest position
  if (r.runs == 1) {
    const int cnt = c->pool_count[seq[0]];
    return cnt == 0 || c->ref_before[r.max_pos] > cnt;
  }
  for (int i = 0; i < n; ++i) {
    const int cnt = c->pool_count[seq[i]];
    if (cnt == 0 || c->ref_before[pos[i]] > cnt) return true;
  }
  return false;
}

// The first row that breaks a precondition of rkv_compress, as an error.
rkv_status compress_row_error(const rkv_ctx* c, const int32_t* src_rows, const int32_t* seq,
                              const int32_t* pos, int n) {
  const rkv::Dims& d = c->d;
  for (int i = 0; i < n; ++i) {
    const int s = seq[i], p = pos[i];
    const int src = src_rows ? src_rows[i] : i;
    if (s < 0 || s >= d.B) return fail(RKV_EINVAL, "row %d: seq %d out of range", i, s);
    if (p < 0 || p >= d.T_cap) return fail(RKV_EINVAL, "row %d: pos %d out of range", i, p);
    if (src < 0) return fail(RKV_EINVAL, "row %d: negative source row", i);
    if (c->ref_before[p + 1] != c->ref_before[p])
      return fail(RKV_EINVAL, "row %d: pos %d is a reference position", i, p);
    if (c->pool_count[s] == 0) return fail(RKV_EEMPTYPOOL, "row %d: seq %d has no reference", i, s);
    // every reference position below p must be in the pool
    if (c->ref_before[p] > c->pool_count[s])
      return fail(RKV_EINVAL, "row %d: references of seq %d before pos %d are not all appended", i,
                  s, p);
  }
  return fail(RKV_EINVAL, "invalid rows");
}

// Per-row plan entries of one tile's rows: retrieval slots q0 .. q0 + cnt - 1 take the
// pass's rows given by `rows`, or r_first .. r_first + cnt - 1 when `rows` is null, of
// sequence s.  The source rows (all the query gather needs) are filled first, so that
// the gather can start while the rest of the plan is built.
void fill_tile_src(int32_t* h, const rkv::PassPlan& p, const int32_t* src_rows, const int* rows,
                   int r_first, int cnt, int q0) {
  int32_t* __restrict__ qsrc = h + p.off_q_src + q0;
  if (!rows) {
    if (src_rows)
      std::memcpy(qsrc, src_rows + r_first, sizeof(int32_t) * cnt);
    else
      for (int r = 0; r < cnt; ++r) qsrc[r] = r_first + r;
  } else {
    for (int r = 0; r < cnt; ++r) qsrc[r] = src_rows ? src_rows[rows[r]] : rows[r];
  }
}

// Positions and storage rows of the same tile rows; returns their largest position (at
// least 1).
int fill_tile_pos(int32_t* h, const rkv::PassPlan& p, const rkv::Dims& d, const int32_t* pos,
                  const int* rows, int r_first, int cnt, int q0, int s) {
  int32_t* __restrict__ qpos = h + p.off_q_pos + q0;
  int32_t* __restrict__ qdst = h + p.off_q_dst + q0;
  const int64_t sT = (int64_t)s * d.T_cap;
  int maxpos = 1;
  for (int r = 0; r < cnt; ++r) {
    const int pr = rows ? pos[rows[r]] : pos[r_first + r];
    maxpos = pr > maxpos ? pr : maxpos;
    qpos[r] = pr;
    qdst[r] = (int32_t)(sT + pr);
  }
  return maxpos;
}

}  // namespace

extern "C" {

const char* rkv_last_error(void) { return g_err.c_str(); }

rkv_status rkv_reference_positions(const rkv_config* cfg, int32_t* pos, int32_t capacity,
                                   int32_t* count) {
  if (!count) return fail(RKV_EINVAL, "count is NULL");
  if (capacity < 0 || (capacity > 0 && !pos)) return fail(RKV_EINVAL, "bad pos / capacity");
  Dims d;
  const rkv_status st = derive(cfg, &d);
  if (st != RKV_OK) return st;
  int32_t n = 0;
  walk_schedule(d.T_cap, d.stride, d.alpha, d.sink, [&](int p) {
    if (n < capacity) pos[n] = p;
    ++n;
  });
  *count = n;
  return RKV_OK;
}

rkv_status rkv_storage_bytes(const rkv_config* cfg, size_t sizes[6]) {
  Dims d;
  rkv_status st = derive(cfg, &d);
  if (st != RKV_OK) return st;
  const size_t pool_rows = (size_t)d.B * d.R_cap, tok_rows = (size_t)d.B * d.T_cap;
  sizes[0] = pool_rows * d.dkv;                 // pool_fp8
  sizes[1] = pool_rows * 4;                     // pool_norm2
  sizes[2] = pool_rows * 4;                     // pool_pos
  sizes[3] = tok_rows * d.code_bytes;           // codes
  sizes[4] = tok_rows * d.G * 4;                // meta
  sizes[5] = tok_rows * d.topk * 4;             // ref_idx
  return RKV_OK;
}

rkv_status rkv_create(const rkv_config* cfg, const void* Wc1, const void* Wc2, const void* Wc3,
                      const void* Wd, const rkv_storage* st, void* stream, rkv_ctx** out) {
  if (!out) return fail(RKV_EINVAL, "out is NULL");
  *out = nullptr;
  Dims d;
  rkv_status r = derive(cfg, &d);
  if (r != RKV_OK) return r;
  if (!st || !Wc1 || !Wc2 || !Wc3 || !Wd) return fail(RKV_EINVAL, "NULL weight or storage");
  const void* ptrs[] = {Wc1, Wc2, Wc3, Wd, st->pool_fp8, st->pool_norm2,
                        st->pool_pos, st->codes, st->meta, st->ref_idx};
  for (const void* p : ptrs) {
    if (!p) return fail(RKV_EINVAL, "NULL storage pointer");
    if (!aligned16(p)) return fail(RKV_EALIGN, "weights and storage must be 16-byte aligned");
  }
  if (!get_encoder()) return fail(RKV_ECUDA, "cuTensorMapEncodeTiled is unavailable");
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  rkv_ctx* c = new rkv_ctx();
  c->cfg = *cfg;
  c->d = d;
  c->st = *st;
  CUDA_OK(cudaGetDevice(&c->device));
  CUDA_OK(cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device));
  c->max_rows = cfg->max_rows > 0 ? cfg->max_rows : 32768;
  c->max_rows = (c->max_rows + kTileM - 1) / kTileM * kTileM;
  c->m_cap = c->max_rows + kTileM * std::min(d.B, c->max_rows);
  c->tiles_cap = c->m_cap / kTileM;
  c->units_cap = c->tiles_cap * ((d.R_cap + kRefTile - 1) / kRefTile);
  c->plan_ints = std::max(4 * c->m_cap + 4 * c->tiles_cap + 2 * c->units_cap + 2 * c->max_rows,
                          4 * c->max_rows);
  c->pool_count.assign(d.B, 0);
  c->ref_before.assign((size_t)d.T_cap + 1, 0);
  walk_schedule(d.T_cap, d.stride, d.alpha, d.sink, [&](int p) { c->ref_before[p + 1] = 1; });
  for (int p = 0; p < d.T_cap; ++p) c->ref_before[p + 1] += c->ref_before[p];

  auto alloc = [&](void** p, size_t bytes) -> cudaError_t { return cudaMalloc(p, bytes); };
  rkv_status fail_status = RKV_OK;
#define ALLOC(ptr, bytes)                                                                 \
  if (fail_status == RKV_OK && alloc(reinterpret_cast<void**>(&(ptr)), (bytes)) != cudaSuccess) \
    fail_status = fail(RKV_ECUDA, "cudaMalloc of %zu bytes failed", (size_t)(bytes));
  ALLOC(c->pool_bf16, (size_t)d.B * d.R_cap * d.dkv * 2);
  ALLOC(c->w12, (size_t)2 * d.dff * d.dkv * 2);
  ALLOC(c->w3, (size_t)d.dc * d.dff * 2);
  ALLOC(c->wd, (size_t)d.dkv * d.dc * 2);
  ALLOC(c->rope_lo, (size_t)kRopeLo * (d.D / 2) * sizeof(float2));
  ALLOC(c->rope_hi, (size_t)d.n_hi * (d.D / 2) * sizeof(float2));
  ALLOC(c->ref_before_dev, ((size_t)d.T_cap + 1) * sizeof(int32_t));
  ALLOC(c->Q, (size_t)c->m_cap * d.parts * d.dkv * 2);
  ALLOC(c->M, (size_t)c->m_cap * d.dkv * 2);
  if (d.B > 1) ALLOC(c->Qd, (size_t)c->max_rows * d.dkv * 2);
  ALLOC(c->H, (size_t)2 * c->m_cap * d.dff * 2);
  ALLOC(c->part, (size_t)c->units_cap * kTileM * 4 * sizeof(int2));
  ALLOC(c->attn_ws, sizeof(float) * kAttnMaxChunks * kAttnMaxGroup * d.N * (2 + d.D));
  ALLOC(c->attn_count, sizeof(int) * d.N);
  {
    const int64_t toks = (int64_t)d.B * d.T_cap < kAttnMaxTokens ? (int64_t)d.B * d.T_cap : kAttnMaxTokens;
    const int64_t tiles = (toks + kTileM - 1) / kTileM;
    ALLOC(c->fa_ws, sizeof(float) * (size_t)tiles * kAttnMaxGroup * d.N * (2 + d.D));
  }
  ALLOC(c->plan_dev[0], (size_t)c->plan_ints * 4);
  ALLOC(c->plan_dev[1], (size_t)c->plan_ints * 4);
  // P: the pool's rows rounded up to whole 128-row tiles, then one zero row
  const size_t p_rows = ((size_t)d.B * d.R_cap + kTileM - 1) / kTileM * kTileM + 1;
  if (d.mean_pre) ALLOC(c->P, p_rows * 2 * d.dff * sizeof(float));
  ALLOC(c->status, 512);
#undef ALLOC
  if (fail_status != RKV_OK) {
    rkv_free(c);
    return fail_status;
  }
  for (int b = 0; b < 2; ++b) {
    if (cudaHostAlloc(reinterpret_cast<void**>(&c->plan_host[b]), (size_t)c->plan_ints * 4,
                      cudaHostAllocMapped) != cudaSuccess ||
        cudaEventCreateWithFlags(&c->plan_copied[b], cudaEventDisableTiming) != cudaSuccess) {
      rkv_free(c);
      return fail(RKV_ECUDA, "pinned staging allocation failed");
    }
    // the device-side address of the mapped buffer; without one, uploads use memcpy
    void* dp = nullptr;
    if (cudaHostGetDevicePointer(&dp, c->plan_host[b], 0) == cudaSuccess && dp != nullptr &&
        (reinterpret_cast<uintptr_t>(dp) & 15u) == 0)
      c->plan_host_dev[b] = static_cast<const int32_t*>(dp);
    else
      cudaGetLastError();
  }

  // RoPE tables in float64, rounded once to fp32: (cos, sin) of l*theta_j and of
  // h*512*theta_j with theta_j = base^(-2j/D).
  {
    const int half = d.D / 2;
    std::vector<float2> lo((size_t)kRopeLo * half), hi((size_t)d.n_hi * half);
    for (int j = 0; j < half; ++j) {
      const double theta = std::pow(cfg->rope_base, -2.0 * j / d.D);
      for (int l = 0; l < kRopeLo; ++l) {
        const double a = (double)l * theta;
        lo[(size_t)l * half + j] = make_float2((float)std::cos(a), (float)std::sin(a));
      }
      for (int h = 0; h < d.n_hi; ++h) {
        const double a = (double)h * kRopeLo * theta;
        hi[(size_t)h * half + j] = make_float2((float)std::cos(a), (float)std::sin(a));
      }
    }
    if (cudaMemcpy(c->rope_lo, lo.data(), lo.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(c->rope_hi, hi.data(), hi.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(c->ref_before_dev, c->ref_before.data(), c->ref_before.size() * sizeof(int32_t),
                   cudaMemcpyHostToDevice) != cudaSuccess) {
      rkv_free(c);
      return fail(RKV_ECUDA, "RoPE or schedule table upload failed");
    }
  }

  // Tensor maps over fixed addresses.
  const uint64_t dkv = d.dkv;
  bool ok = true;
  ok &= make_map(&c->tm_q, c->Q, (uint64_t)d.parts * dkv, c->m_cap, (uint64_t)d.parts * dkv * 2, kTileM);
  ok &= make_map(&c->tm_pool, c->pool_bf16, dkv, (uint64_t)d.B * d.R_cap, dkv * 2, kRefTile);
  ok &= make_map(&c->tm_qa, c->Q, dkv, c->m_cap, (uint64_t)d.parts * dkv * 2, kTileM / 2);
  ok &= make_map(&c->tm_m, c->M, dkv, c->m_cap, dkv * 2, kTileM / 2);
  if (c->Qd) ok &= make_map(&c->tm_qd, c->Qd, dkv, c->max_rows, dkv * 2, kTileM / 2);
  ok &= make_map(&c->tm_w12, c->w12, dkv, (uint64_t)2 * d.dff, dkv * 2, kEncN);
  ok &= make_map(&c->tm_h3, c->H, (uint64_t)2 * d.dff, c->m_cap, (uint64_t)2 * d.dff * 2, kTileM);
  const uint32_t bn3 = d.dc % 256 == 0 ? 256u : (d.dc % 128 == 0 ? 128u : 64u);
  ok &= make_map(&c->tm_w3, c->w3, d.dff, d.dc, (uint64_t)d.dff * 2, bn3);
  if (d.dc % 128 == 0)
    ok &= make_map(&c->tm_w3_128, c->w3, d.dff, d.dc, (uint64_t)d.dff * 2, 128u);
  ok &= make_map(&c->tm_wd, c->wd, d.dc, dkv, (uint64_t)d.dc * 2, kDecN);
  if (d.mean_pre) {
    ok &= make_map(&c->tm_pool128, c->pool_bf16, dkv, (uint64_t)d.B * d.R_cap, dkv * 2, kTileM);
    ok &= make_map(&c->tm_qa128, c->Q, dkv, c->m_cap, (uint64_t)d.parts * dkv * 2, kTileM);
    if (c->Qd) ok &= make_map(&c->tm_qd128, c->Qd, dkv, c->max_rows, dkv * 2, kTileM);
  }
  if (!ok) {
    rkv_free(c);
    return fail(RKV_ECUDA, "cuTensorMapEncodeTiled rejected a tensor map");
  }

  c->zero_line = reinterpret_cast<const uint8_t*>(c->status) + 256;
  cudaError_t e = cudaMemsetAsync(c->status, 0, 512, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->Q, 0, (size_t)c->m_cap * d.parts * d.dkv * 2, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->M, 0, (size_t)c->m_cap * d.dkv * 2, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->pool_bf16, 0, (size_t)d.B * d.R_cap * d.dkv * 2, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->H, 0, (size_t)2 * c->m_cap * d.dff * 2, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->attn_count, 0, sizeof(int) * d.N, s);
  if (e == cudaSuccess && c->P) e = cudaMemsetAsync(c->P, 0, p_rows * 2 * d.dff * sizeof(float), s);
  if (e == cudaSuccess) e = launch_init_storage(c, s);
  if (e == cudaSuccess)
    e = launch_repack_weights(c, static_cast<const __nv_bfloat16*>(Wc1),
                              static_cast<const __nv_bfloat16*>(Wc2),
                              static_cast<const __nv_bfloat16*>(Wc3),
                              static_cast<const __nv_bfloat16*>(Wd), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    rkv_free(c);
    return fail(RKV_ECUDA, "initialisation failed: %s", cudaGetErrorString(e));
  }
  *out = c;
  return RKV_OK;
}

rkv_status rkv_pool_append(rkv_ctx* c, const void* kv, int64_t kv_row_stride,
                           const int32_t* src_rows, const int32_t* seq, const int32_t* pos,
                           int32_t n, void* stream) {
  if (!c) return fail(RKV_EINVAL, "ctx is NULL");
  if (n < 0) return fail(RKV_EINVAL, "n < 0");
  if (n == 0) return RKV_OK;
  if (!kv || !seq || !pos) return fail(RKV_EINVAL, "NULL kv, seq or pos");
  if (!aligned16(kv)) return fail(RKV_EALIGN, "kv must be 16-byte aligned");
  const Dims& d = c->d;
  if (kv_row_stride < d.dkv || kv_row_stride % 8 != 0)
    return fail(RKV_EINVAL, "kv_row_stride must be >= 2*d_k and a multiple of 8");
  // validate everything before touching the host mirror: one branch-free pass for the
  // usual call, the row-by-row pass (which names the first bad row) otherwise
  std::vector<int32_t> next(c->pool_count);
  const bool fast = append_rows_ok_one_seq(c, src_rows, seq, pos, n);
  if (fast) next[seq[0]] += n;
  for (int i = 0; i < n && !fast; ++i) {
    const int s = seq[i], p = pos[i];
    const int src = src_rows ? src_rows[i] : i;
    if (s < 0 || s >= d.B) return fail(RKV_EINVAL, "row %d: seq %d out of range", i, s);
    if (p < 0 || p >= d.T_cap) return fail(RKV_EINVAL, "row %d: pos %d out of range", i, p);
    if (src < 0) return fail(RKV_EINVAL, "row %d: negative source row", i);
    const int slot = c->ref_before[p];
    if (c->ref_before[p + 1] == slot)
      return fail(RKV_EINVAL, "row %d: pos %d is not a reference position", i, p);
    if (slot >= d.R_cap) return fail(RKV_ECAPACITY, "row %d: slot %d >= max_refs", i, slot);
    if (slot != next[s])
      return fail(RKV_EINVAL, "row %d: seq %d expects its reference slot %d next, got pos %d (slot %d)",
                  i, s, next[s], p, slot);
    next[s] = slot + 1;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int r0 = 0; r0 < n; r0 += c->max_rows) {
    const int m = std::min(c->max_rows, n - r0);
    int b;
    int32_t* h = staging_acquire(c, &b);
    for (int i = 0; i < m; ++i) {
      const int k = r0 + i;
      const int s = seq[k], p = pos[k];
      h[4 * i + 0] = src_rows ? src_rows[k] : k;
      h[4 * i + 1] = s * d.R_cap + c->ref_before[p];
      h[4 * i + 2] = p;
      h[4 * i + 3] = s * d.T_cap + p;
    }
    // with mean_precompute, the pool tiles (128 slots) these references fall in, in
    // increasing order, follow the rows in the plan
    int n_pt = 0;
    if (d.mean_pre) {
      int last = -1;
      bool sorted = true;
      for (int i = 0; i < m; ++i) {
        const int t = h[4 * i + 1] / kTileM;
        if (t != last) {
          if (t < last) sorted = false;
          h[4 * m + n_pt++] = t;
          last = t;
        }
      }
      if (!sorted) {
        std::sort(h + 4 * m, h + 4 * m + n_pt);
        n_pt = (int)(std::unique(h + 4 * m, h + 4 * m + n_pt) - (h + 4 * m));
      }
    }
    if (4 * m + n_pt > c->plan_ints) return fail(RKV_ECAPACITY, "append plan exceeds the staging buffer");
    CUDA_OK(staging_upload(c, b, 0, 4 * m + n_pt, st));
    CUDA_OK(launch_pool_append(c, kv, kv_row_stride, c->plan_dev[b], m, st));
    if (n_pt) CUDA_OK(launch_pool_preact(c, c->plan_dev[b] + 4 * m, n_pt, st));
  }
  c->pool_count = next;
  return RKV_OK;
}

rkv_status rkv_compress(rkv_ctx* c, const void* kv, int64_t kv_row_stride, const int32_t* src_rows,
                        const int32_t* seq, const int32_t* pos, int32_t n, void* stream) {
  if (!c) return fail(RKV_EINVAL, "ctx is NULL");
  if (n < 0) return fail(RKV_EINVAL, "n < 0");
  if (n == 0) return RKV_OK;
  if (!kv || !seq || !pos) return fail(RKV_EINVAL, "NULL kv, seq or pos");
  if (!aligned16(kv)) return fail(RKV_EALIGN, "kv must be 16-byte aligned");
  const Dims& d = c->d;
  if (kv_row_stride < d.dkv || kv_row_stride % 8 != 0)
    return fail(RKV_EINVAL, "kv_row_stride must be >= 2*d_k and a multiple of 8");
  // one branch-free pass over the rows; the row-by-row pass that names the first bad
  // row runs only when it found one
  const int32_t* rb = c->ref_before.data();
  const RowScan scan = !d.fixed                          ? scan_compress_rows<2>(d, rb, src_rows, seq, pos, n)
                       : (d.stride & (d.stride - 1)) == 0 ? scan_compress_rows<0>(d, rb, src_rows, seq, pos, n)
                                                          : scan_compress_rows<1>(d, rb, src_rows, seq, pos, n);
  if (scan.bad || compress_pools_bad(c, scan, seq, pos, n))
    return compress_row_error(c, src_rows, seq, pos, n);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::vector<int> order, gbeg;
  std::vector<int32_t> tseq, trow0, tnrt;
  for (int r0 = 0; r0 < n; r0 += c->max_rows) {
    const int m = std::min(c->max_rows, n - r0);
    // ---- plan: rows grouped by sequence (stable), each group padded to 128 rows.  A
    // counting sort by sequence id (O(m + B)); nothing to do when the ids never decrease.
    bool grouped = scan.grouped;
    if (!grouped) {
      unsigned dec = 0;
      for (int i = 1; i < m; ++i) dec |= (unsigned)(seq[r0 + i] < seq[r0 + i - 1]);
      grouped = dec == 0;
    }
    const int* ord = nullptr;                          // group order; null: rows as given
    if (!grouped) {
      order.resize(m);
      std::vector<int> start(d.B + 1, 0);
      for (int i = 0; i < m; ++i) ++start[seq[r0 + i] + 1];
      for (int b2 = 0; b2 < d.B; ++b2) start[b2 + 1] += start[b2];
      for (int i = 0; i < m; ++i) order[start[seq[r0 + i]]++] = r0 + i;
      ord = order.data();
    }
    // group boundaries (positions in group order), padded sizes
    gbeg.clear();
    int m_pad = 0, ntiles = 0;
    if (scan.runs == 1) {
      gbeg.push_back(0);
      m_pad = (m + kTileM - 1) / kTileM * kTileM;
      ntiles = m_pad / kTileM;
    } else {
      int i = 0;
      int si = seq[ord ? ord[0] : r0];
      for (int j = 1; j <= m; ++j) {
        const int sj = j < m ? seq[ord ? ord[j] : r0 + j] : -1;
        if (sj == si) continue;
        gbeg.push_back(i);
        const int padded = (j - i + kTileM - 1) / kTileM * kTileM;
        m_pad += padded;
        ntiles += padded / kTileM;
        i = j;
        si = sj;
      }
    }
    gbeg.push_back(m);
    // plan layout: per-row arrays first, then tiles, then units (counted while filling)
    PassPlan p;
    p.n_rows = m;
    p.m_pad = m_pad;
    p.n_tiles = ntiles;
    p.off_q_src = 0;
    p.off_q_pos = m_pad;
    p.off_q_dst = 2 * m_pad;
    p.off_t_seq = 3 * m_pad;
    p.off_t_row0 = p.off_t_seq + ntiles;
    p.off_t_nrt = p.off_t_row0 + ntiles;
    p.off_t_u0 = p.off_t_nrt + ntiles;
    p.off_u_tile = p.off_t_u0 + ntiles;
    if (m_pad > c->m_cap || p.off_u_tile > c->plan_ints)
      return fail(RKV_ECAPACITY, "compress pass exceeds the planned scratch");
    int b;
    int32_t* h = staging_acquire(c, &b);
    // the query rows' sources first: upload them and start the query gather
    for (size_t g = 0, q = 0; g + 1 < gbeg.size(); ++g) {
      const int i = gbeg[g], j = gbeg[g + 1];
      const int padded = (j - i + kTileM - 1) / kTileM * kTileM;
      fill_tile_src(h, p, src_rows, ord ? ord + i : nullptr, r0 + i, j - i, (int)q);
      for (int k = j - i; k < padded; ++k) h[p.off_q_src + q + k] = -1;
      q += padded;
    }
    CUDA_OK(staging_upload(c, b, p.off_q_src, m_pad, st));
    const int32_t* plan = c->plan_dev[b];
    CUDA_OK(launch_prep_queries(c, kv, kv_row_stride, plan + p.off_q_src, p.m_pad, st));
    tseq.clear();
    trow0.clear();
    tnrt.clear();
    int q = 0, n_units = 0;
    for (size_t g = 0; g + 1 < gbeg.size(); ++g) {
      const int i = gbeg[g], j = gbeg[g + 1];
      const int s = seq[ord ? ord[i] : r0 + i];
      for (int k = i; k < j; k += kTileM) {
        const int kend = std::min(j, k + kTileM);
        const int maxpos = fill_tile_pos(h, p, d, pos, ord ? ord + k : nullptr, r0 + k, kend - k,
                                         q + (k - i), s);
        const int nrt = (c->ref_before[maxpos] + kRefTile - 1) / kRefTile;
        tseq.push_back(s);
        trow0.push_back(q + (k - i));
        tnrt.push_back(nrt);
        n_units += nrt;
      }
      const int padded = (j - i + kTileM - 1) / kTileM * kTileM;
      for (int k = j - i; k < padded; ++k) {
        h[p.off_q_pos + q + k] = -1;
        h[p.off_q_dst + q + k] = -1;
      }
      q += padded;
    }
    p.n_units = n_units;
    p.off_u_rt = p.off_u_tile + n_units;
    p.total_ints = p.off_u_rt + n_units;
    // several sequences in the pass: the encoder GEMMs take its rows densely packed
    p.dense = gbeg.size() > 2;
    if (p.dense) {
      p.off_q_comp = p.total_ints;
      p.off_d_src = p.off_q_comp + m_pad;
      p.off_d_dst = p.off_d_src + m;
      p.total_ints = p.off_d_dst + m;
    }
    if (n_units > c->units_cap || p.total_ints > c->plan_ints || (p.dense && !c->Qd))
      return fail(RKV_ECAPACITY, "compress pass exceeds the planned retrieval scratch");
    if (p.dense) {
      // dense row j = the j-th row in group order; retrieval row q of group g sits at
      // the group's padded offset
      for (size_t g = 0, q = 0; g + 1 < gbeg.size(); ++g) {
        const int i = gbeg[g], j = gbeg[g + 1];
        const int padded = (j - i + kTileM - 1) / kTileM * kTileM;
        for (int k = 0; k < padded; ++k) {
          const bool real = k < j - i;
          h[p.off_q_comp + q + k] = real ? i + k : -1;
          if (real) {
            h[p.off_d_src + i + k] = h[p.off_q_src + q + k];
            h[p.off_d_dst + i + k] = h[p.off_q_dst + q + k];
          }
        }
        q += padded;
      }
    }
    // tiles in order; units tile-major, pool tiles in increasing slot order
    int u = 0;
    for (int i = 0; i < ntiles; ++i) {
      h[p.off_t_seq + i] = tseq[i];
      h[p.off_t_row0 + i] = trow0[i];
      h[p.off_t_nrt + i] = tnrt[i];
      h[p.off_t_u0 + i] = u;
      for (int rt = 0; rt < tnrt[i]; ++rt, ++u) {
        h[p.off_u_tile + u] = i;
        h[p.off_u_rt + u] = rt;
      }
    }
    CUDA_OK(staging_upload(c, b, p.off_q_pos, p.total_ints - p.off_q_pos, st));
    if (p.dense) CUDA_OK(launch_prep_dense(c, kv, kv_row_stride, plan + p.off_d_src, m, st));
    CUDA_OK(launch_retrieve(c, p, plan, st));
    CUDA_OK(launch_retrieve_merge(c, p, plan, st));
    if (!d.mean_pre) CUDA_OK(launch_mean_rows(c, p, plan, st));
    CUDA_OK(launch_gemm12(c, p, plan, st));
    CUDA_OK(launch_gemm3_quant(c, p, plan, st));
  }
  return RKV_OK;
}

rkv_status rkv_reconstruct(rkv_ctx* c, const int32_t* seq, const int32_t* pos, int32_t n_sel,
                           void* k_out, void* v_out, void* stream) {
  if (!c) return fail(RKV_EINVAL, "ctx is NULL");
  if (n_sel < 0) return fail(RKV_EINVAL, "n_sel < 0");
  if (n_sel == 0) return RKV_OK;
  if (!seq || !pos || !k_out || !v_out) return fail(RKV_EINVAL, "NULL seq, pos or output");
  // the kernel writes whole 32-byte sectors
  if ((reinterpret_cast<uintptr_t>(k_out) & 31u) || (reinterpret_cast<uintptr_t>(v_out) & 31u) ||
      (reinterpret_cast<uintptr_t>(seq) & 3u) || (reinterpret_cast<uintptr_t>(pos) & 3u))
    return fail(RKV_EALIGN, "outputs must be 32-byte aligned, seq/pos 4-byte aligned");
  CUDA_OK(launch_reconstruct(c, seq, pos, n_sel, k_out, v_out, static_cast<cudaStream_t>(stream)));
  return RKV_OK;
}

rkv_status rkv_reconstruct_multi(rkv_ctx* const* ctxs, int32_t n, const int32_t* const* seq,
                                 const int32_t* const* pos, const int32_t* n_sel,
                                 void* const* k_out, void* const* v_out, void* stream) {
  if (!ctxs || !seq || !pos || !n_sel || !k_out || !v_out)
    return fail(RKV_EINVAL, "NULL argument array");
  if (n < 1 || n > kReconMaxProblems)
    return fail(RKV_EINVAL, "n must be in [1, %d]", kReconMaxProblems);
  const rkv_ctx* c0 = ctxs[0];
  if (!c0) return fail(RKV_EINVAL, "ctxs[0] is NULL");
  const Dims& d = c0->d;
  for (int i = 0; i < n; ++i) {
    const rkv_ctx* c = ctxs[i];
    if (!c) return fail(RKV_EINVAL, "ctxs[%d] is NULL", i);
    const Dims& e = c->d;
    // one kernel serves all: every dimension, format and table must agree
    if (c->device != c0->device || e.N != d.N || e.D != d.D || e.dc != d.dc || e.topk != d.topk ||
        e.bits != d.bits || e.B != d.B || e.T_cap != d.T_cap || e.R_cap != d.R_cap ||
        e.out_f32 != d.out_f32 || c->cfg.rope_base != c0->cfg.rope_base)
      return fail(RKV_EINVAL, "ctxs[%d] differs from ctxs[0] in device, shape, format or tables", i);
    if (n_sel[i] < 0) return fail(RKV_EINVAL, "n_sel[%d] < 0", i);
    if (n_sel[i] == 0) continue;
    if (!seq[i] || !pos[i] || !k_out[i] || !v_out[i])
      return fail(RKV_EINVAL, "NULL seq, pos or output of problem %d", i);
    if ((reinterpret_cast<uintptr_t>(k_out[i]) & 31u) || (reinterpret_cast<uintptr_t>(v_out[i]) & 31u) ||
        (reinterpret_cast<uintptr_t>(seq[i]) & 3u) || (reinterpret_cast<uintptr_t>(pos[i]) & 3u))
      return fail(RKV_EALIGN, "problem %d: outputs must be 32-byte aligned, seq/pos 4-byte aligned", i);
  }
  // one problem with tokens: the single restore (its ranges are balanced for one problem)
  int live = 0, only = -1;
  for (int i = 0; i < n; ++i)
    if (n_sel[i] > 0) ++live, only = i;
  if (live == 0) return RKV_OK;
  if (live == 1) {
    CUDA_OK(launch_reconstruct(const_cast<rkv_ctx*>(ctxs[only]), seq[only], pos[only], n_sel[only],
                               k_out[only], v_out[only], static_cast<cudaStream_t>(stream)));
    return RKV_OK;
  }
  CUDA_OK(launch_reconstruct_multi(const_cast<rkv_ctx* const*>(ctxs), n, seq, pos, n_sel, k_out,
                                   v_out, static_cast<cudaStream_t>(stream)));
  return RKV_OK;
}

rkv_status rkv_sparse_attention(rkv_ctx* c, const float* q, int32_t n_q_heads, const void* k,
                                const void* v, int32_t n, float* out, void* stream) {
  if (!c) return fail(RKV_EINVAL, "ctx is NULL");
  if (!q || !k || !v || !out) return fail(RKV_EINVAL, "NULL q, k, v or out");
  const Dims& d = c->d;
  if (n_q_heads < d.N || n_q_heads % d.N != 0 || n_q_heads / d.N > kAttnMaxGroup)
    return fail(RKV_EINVAL, "n_q_heads must be a multiple of n_kv_heads, at most %d times it",
                kAttnMaxGroup);
  if (n < 1 || n > kAttnMaxTokens)
    return fail(RKV_EINVAL, "n must be in [1, %d] (softmax over the selected tokens)",
                kAttnMaxTokens);
  if ((reinterpret_cast<uintptr_t>(k) & 15u) || (reinterpret_cast<uintptr_t>(v) & 15u) ||
      (reinterpret_cast<uintptr_t>(q) & 3u) || (reinterpret_cast<uintptr_t>(out) & 3u))
    return fail(RKV_EALIGN, "k and v must be 16-byte aligned, q and out 4-byte aligned");
  CUDA_OK(launch_attention(c, q, n_q_heads, k, v, n, out, static_cast<cudaStream_t>(stream)));
  return RKV_OK;
}

rkv_status rkv_restore_attend(rkv_ctx* c, const int32_t* seq, const int32_t* pos, int32_t n_sel,
                              const float* q, int32_t n_q_heads, float* out, void* stream) {
  if (!c) return fail(RKV_EINVAL, "ctx is NULL");
  if (!seq || !pos || !q || !out) return fail(RKV_EINVAL, "NULL seq, pos, q or out");
  const Dims& d = c->d;
  if (d.D != 128 || d.out_f32)
    return fail(RKV_EINVAL, "the fused restore + attention needs head_dim 128 and bf16 outputs");
  if (n_q_heads < d.N || n_q_heads % d.N != 0 || n_q_heads / d.N > kAttnMaxGroup)
    return fail(RKV_EINVAL, "n_q_heads must be a multiple of n_kv_heads, at most %d times it",
                kAttnMaxGroup);
  if (n_sel < 1 || n_sel > kAttnMaxTokens || (int64_t)n_sel > (int64_t)d.B * d.T_cap)
    return fail(RKV_EINVAL, "n_sel must be in [1, min(%d, B * max_tokens)]", kAttnMaxTokens);
  if ((reinterpret_cast<uintptr_t>(q) & 7u) || (reinterpret_cast<uintptr_t>(out) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq) & 3u) || (reinterpret_cast<uintptr_t>(pos) & 3u))
    return fail(RKV_EALIGN, "q must be 8-byte aligned, out, seq and pos 4-byte aligned");
  CUDA_OK(launch_restore_attend(c, seq, pos, n_sel, q, n_q_heads, out,
                                static_cast<cudaStream_t>(stream)));
  return RKV_OK;
}

rkv_status rkv_pool_cache(rkv_ctx* c, void** ptr, size_t* bytes) {
  if (!c || !ptr || !bytes) return fail(RKV_EINVAL, "NULL argument");
  *ptr = c->pool_bf16;
  *bytes = (size_t)c->d.B * c->d.R_cap * c->d.dkv * 2;
  return RKV_OK;
}

rkv_status rkv_reset(rkv_ctx* c, int32_t seq, void* stream) {
  if (!c) return fail(RKV_EINVAL, "ctx is NULL");
  if (seq < -1 || seq >= c->d.B) return fail(RKV_EINVAL, "seq %d out of range", seq);
  CUDA_OK(launch_init_storage(c, static_cast<cudaStream_t>(stream), seq));
  if (seq < 0)
    std::fill(c->pool_count.begin(), c->pool_count.end(), 0);
  else
    c->pool_count[seq] = 0;
  return RKV_OK;
}

rkv_status rkv_get_status(rkv_ctx* c, int32_t* flags, void* stream) {
  if (!c || !flags) return fail(RKV_EINVAL, "NULL ctx or flags");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  CUDA_OK(cudaMemcpyAsync(&v, c->status, 4, cudaMemcpyDeviceToHost, s));
  CUDA_OK(cudaMemsetAsync(c->status, 0, 4, s));
  CUDA_OK(cudaStreamSynchronize(s));
  *flags = v;
  if (v == 0) return RKV_OK;
  if (v & RKV_FLAG_TIMEOUT) return fail(RKV_ETIMEOUT, "a kernel wait timed out (flags 0x%x)", v);
  return fail(RKV_EDEVICE, "device status flags 0x%x", v);
}

void rkv_free(rkv_ctx* c) {
  if (!c) return;
  cudaFree(c->pool_bf16);
  cudaFree(c->w12);
  cudaFree(c->attn_ws);
  cudaFree(c->attn_count);
  cudaFree(c->fa_ws);
  cudaFree(c->P);
  cudaFree(c->w3);
  cudaFree(c->wd);
  cudaFree(c->rope_lo);
  cudaFree(c->rope_hi);
  cudaFree(c->ref_before_dev);
  cudaFree(c->Q);
  cudaFree(c->M);
  cudaFree(c->Qd);
  cudaFree(c->H);
  cudaFree(c->part);
  cudaFree(c->status);
  for (int b = 0; b < 2; ++b) {
    cudaFree(c->plan_dev[b]);
    if (c->plan_host[b]) cudaFreeHost(c->plan_host[b]);
    if (c->plan_copied[b]) cudaEventDestroy(c->plan_copied[b]);
  }
  for (auto& t : c->timings)
    for (cudaEvent_t e : t.pending) cudaEventDestroy(e);
  delete c;
}

rkv_status rkv_set_timing(rkv_ctx* c, int32_t enable) {
  if (!c) return fail(RKV_EINVAL, "ctx is NULL");
  c->timing = enable != 0;
  return RKV_OK;
}

int32_t rkv_get_timing(rkv_ctx* c, rkv_kernel_timing* out, int32_t max_entries, int32_t reset) {
  if (!c) return 0;
  int32_t n = 0;
  for (auto& t : c->timings) {
    for (size_t i = 0; i + 1 < t.pending.size(); i += 2) {
      float ms = 0.f;
      cudaEventSynchronize(t.pending[i + 1]);
      if (cudaEventElapsedTime(&ms, t.pending[i], t.pending[i + 1]) == cudaSuccess) t.total_ms += ms;
      cudaEventDestroy(t.pending[i]);
      cudaEventDestroy(t.pending[i + 1]);
    }
    t.pending.clear();
    if (out && n < max_entries) {
      std::memset(&out[n], 0, sizeof(rkv_kernel_timing));
      std::snprintf(out[n].name, sizeof(out[n].name), "%s", t.name.c_str());
      out[n].launches = t.launches;
      out[n].total_ms = t.total_ms;
    }
    ++n;
  }
  if (reset) c->timings.clear();
  return n;
}

int64_t rkv_launch_count(rkv_ctx* c) { return c ? c->launches : 0; }

rkv_status rkv_debug_timeout_probe(rkv_ctx* c, void* stream) {
  if (!c) return fail(RKV_EINVAL, "ctx is NULL");
  CUDA_OK(launch_timeout_probe(c, static_cast<cudaStream_t>(stream)));
  return RKV_OK;
}

rkv_status rkv_debug_scratch(rkv_ctx* c, int32_t which, void** ptr, size_t* bytes) {
  if (!c || !ptr || !bytes) return fail(RKV_EINVAL, "NULL argument");
  if (which == 0) {
    *ptr = c->M;
    *bytes = (size_t)c->m_cap * c->d.dkv * 2;
  } else if (which == 1) {
    *ptr = c->H;
    *bytes = (size_t)2 * c->m_cap * c->d.dff * 2;
  } else if (which == 2) {
    *ptr = c->Q;
    *bytes = (size_t)c->m_cap * c->d.parts * c->d.dkv * 2;
  } else if (which == 3 && c->P) {
    *ptr = c->P;
    *bytes = (((size_t)c->d.B * c->d.R_cap + kTileM - 1) / kTileM * kTileM) * 2 * c->d.dff * 4;
  } else {
    return fail(RKV_EINVAL, "which must be 0, 1, 2 (or 3 with mean_precompute)");
  }
  return RKV_OK;
}

}  // extern "C"
