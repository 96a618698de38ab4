// rkv_internal.h - context layout and the launchers shared by the host API and kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/rkv.h"

namespace rkv {

constexpr int kTileM = 128;        // rows per tensor-core tile (one TMEM lane per row)
constexpr int kTileK = 64;         // bf16 elements per 128-byte swizzled row
constexpr int kRefTile = 256;      // references per retrieval tile
constexpr int kEncN = 256;         // GEMM-1/2 N tile: 128 W_c1 + 128 W_c2 columns
constexpr int kDecN = 128;         // decoder N tile (one head of D = 128)
constexpr int kRopeLo = 512;       // positions per low RoPE table
constexpr int kReconMaxProblems = 32;   // contexts one rkv_reconstruct_multi launch restores

// Derived sizes of a configuration.
struct Dims {
  int N, D, dk, dkv, dc, dff, topk, group, bits, stride;
  int G;           // groups per token
  int code_bytes;  // bytes of one packed code row
  int B, T_cap, R_cap;
  double alpha;    // dynamic schedule growth (0: fixed stride)
  int sink;        // sink tokens
  int fixed;       // the schedule is pos % stride == 0
  int n_sched;     // schedule positions below T_cap
  int kv_f32, out_f32;
  int mean_pre;    // the mean's pre-activations from the references' (table P)
  int parts;       // 3 bf16 pieces per fp32 query element, 1 for bf16
  int n_hi;        // rows of the high RoPE table
};

// One kernel's accumulated event time (instrumentation).
struct TimingSlot {
  std::string name;
  int64_t launches = 0;
  double total_ms = 0.0;
  std::vector<cudaEvent_t> pending;  // start/stop pairs not yet read
};

// Device plan of one compress pass (int32 arrays inside one buffer).  Retrieval works
// in retrieval order (the pass's rows grouped by sequence, each group padded to 128
// rows, so a tile queries one pool); the encoder GEMMs work on the pass's rows packed
// densely (row j = the j-th row in group order).  With one group the two orders agree
// on the first n_rows rows and the dense arrays are not used.
struct PassPlan {
  int n_rows = 0;      // compact rows (this pass)
  int m_pad = 0;       // retrieval-order rows, padded per sequence to 128
  int n_tiles = 0;     // retrieval tiles (128 query rows of one sequence)
  int n_units = 0;     // retrieval units: (tile, 256-reference pool tile)
  bool dense = false;  // several groups: the encoder reads the dense arrays below
  // offsets (in int32 elements) inside the plan buffer
  int off_q_src, off_q_pos, off_q_dst, off_t_seq, off_t_row0, off_t_nrt, off_t_u0, off_u_tile,
      off_u_rt;
  int off_q_comp = 0;  // [m_pad] dense row of each retrieval row, -1 for padding
  int off_d_src = 0;   // [n_rows] source kv row of each dense row
  int off_d_dst = 0;   // [n_rows] storage row of each dense row
  int total_ints = 0;
};

}  // namespace rkv

struct rkv_ctx {
  rkv_config cfg;
  rkv::Dims d;
  rkv_storage st;
  int device = 0;
  int num_sms = 0;
  int recon_smem = 0;          // dynamic shared memory the restore kernel is set up for
  int max_rows = 0;    // compact rows per pass
  int m_cap = 0;       // retrieval-order rows per pass (with padding)
  int tiles_cap = 0;

  // library-owned device memory
  __nv_bfloat16* pool_bf16 = nullptr;  // [B, R_cap, 2d_k] bf16 copy of the FP8 pool (retrieval
                                       // operand, kept in step by pool_append)
  __nv_bfloat16* w12 = nullptr;   // [2 d_ff, 2d_k]: per 256-row tile, 128 W_c1^T rows then 128 W_c2^T rows
  __nv_bfloat16* w3 = nullptr;    // [d_c, d_ff] = W_c3^T
  __nv_bfloat16* wd = nullptr;    // [2d_k, d_c] = W_d^T
  float2* rope_lo = nullptr;      // [512][D/2] (cos, sin)(l * theta_j)
  float2* rope_hi = nullptr;      // [n_hi][D/2] (cos, sin)(h * 512 * theta_j)
  int32_t* ref_before_dev = nullptr;   // [T_cap + 1] device copy of ref_before
  __nv_bfloat16* Q = nullptr;     // [m_cap, parts * 2d_k] retrieval-order queries
  __nv_bfloat16* M = nullptr;     // [m_cap, 2d_k] bf16 reference means, dense order
  __nv_bfloat16* Qd = nullptr;    // [max_rows, 2d_k] bf16 kv rows in dense order (B > 1 only;
                                  // with one sequence the query rows serve)
  __nv_bfloat16* H = nullptr;     // [m_cap, 2 d_ff] row q: [hi | lo] bf16 parts of the fp32
                                  // hidden difference h(kv_q) - h(mean_q)
  int2* part = nullptr;           // [units_cap, 128, 4] partial top-k (distance bits, slot)
  float* attn_ws = nullptr;       // sparse attention chunk partials (m, l, acc), kAttnMaxChunks
                                  // x kAttnMaxGroup N query heads
  int* attn_count = nullptr;      // [N] finished chunks per key/value head (zero between calls)
  float* fa_ws = nullptr;         // restore + attention partials (m, l, o) per token tile and
                                  // query head: up to kAttnMaxTokens / 128 tiles x 8 N heads
  int fused_smem = 0;             // dynamic shared memory the fused kernel is set up for
  int multi_smem = 0;             // ... and the multi-context restore kernel
  int units_cap = 0;
  int32_t* plan_dev[2] = {nullptr, nullptr};
  int32_t* plan_host[2] = {nullptr, nullptr};   // pinned staging
  const int32_t* plan_host_dev[2] = {nullptr, nullptr};   // its device-side address (mapped)
  cudaEvent_t plan_copied[2] = {nullptr, nullptr};
  int plan_ints = 0;
  int plan_flip = 0;
  float* P = nullptr;             // mean_precompute: [B R_cap rounded up to 128, 2 d_ff] fp32
                                  // r [W_c1 | W_c2] of each pool slot, columns in W12's order
  int* status = nullptr;          // device status word (first 64 bytes of a 512-byte block)
  const uint8_t* zero_line = nullptr;   // 256 zero bytes in the same block (gather source)

  // TMA descriptors (fixed addresses, built once)
  CUtensorMap tm_q, tm_pool, tm_w12, tm_h3, tm_w3, tm_w3_128, tm_wd;
  CUtensorMap tm_qa, tm_m;        // GEMM-1/2 A halves: the bf16 kv piece of Q, and M (64 rows)
  CUtensorMap tm_qd;              // GEMM-1/2 kv half from Qd (dense passes)
  CUtensorMap tm_pool128, tm_qa128, tm_qd128;   // 128-row boxes: mean_precompute GEMMs

  // host mirror of each sequence's pool fill
  std::vector<int32_t> pool_count;
  std::vector<int32_t> ref_before;   // [T_cap + 1]: schedule positions below p

  // instrumentation
  bool timing = false;
  std::vector<rkv::TimingSlot> timings;
  int64_t launches = 0;
};

namespace rkv {

// ---- launchers (defined in the kernel translation units) ----
// Each returns cudaGetLastError() of its launch.
cudaError_t launch_init_storage(rkv_ctx* c, cudaStream_t s, int seq = -1);
cudaError_t launch_repack_weights(rkv_ctx* c, const __nv_bfloat16* Wc1, const __nv_bfloat16* Wc2,
                                  const __nv_bfloat16* Wc3, const __nv_bfloat16* Wd,
                                  cudaStream_t s);
cudaError_t launch_pool_append(rkv_ctx* c, const void* kv, int64_t stride, const int32_t* plan,
                               int n, cudaStream_t s);
cudaError_t launch_prep_queries(rkv_ctx* c, const void* kv, int64_t stride, const int32_t* q_src,
                                int m_pad, cudaStream_t s);
// bf16 kv rows of the dense order into Qd (n rows, sources d_src)
cudaError_t launch_prep_dense(rkv_ctx* c, const void* kv, int64_t stride, const int32_t* d_src,
                              int n, cudaStream_t s);
cudaError_t launch_retrieve(rkv_ctx* c, const PassPlan& p, const int32_t* plan, cudaStream_t s);
cudaError_t launch_retrieve_merge(rkv_ctx* c, const PassPlan& p, const int32_t* plan,
                                  cudaStream_t s);
cudaError_t launch_mean_rows(rkv_ctx* c, const PassPlan& p, const int32_t* plan, cudaStream_t s);
// GEMM-1/2 and the hidden difference; with mean_precompute over kv rows only, the mean's
// hidden row from P (plan: the pass's plan, for each dense row's storage row)
cudaError_t launch_gemm12(rkv_ctx* c, const PassPlan& p, const int32_t* plan, cudaStream_t s);
cudaError_t launch_gemm3_quant(rkv_ctx* c, const PassPlan& p, const int32_t* plan,
                               cudaStream_t s);
// mean_precompute: P rows of the pool tiles listed in `tiles` (128 slots each, indices
// into [B R_cap] rows), from the bf16 pool copy
cudaError_t launch_pool_preact(rkv_ctx* c, const int32_t* tiles, int n_tiles, cudaStream_t s);
cudaError_t launch_reconstruct(rkv_ctx* c, const int32_t* seq, const int32_t* pos, int n_sel,
                               void* k_out, void* v_out, cudaStream_t s);
// One launch restoring the selections of n <= kReconMaxProblems contexts of equal
// dimensions (validated by the caller); the timing slot is the first context's.
cudaError_t launch_reconstruct_multi(rkv_ctx* const* cs, int n, const int32_t* const* seqs,
                                     const int32_t* const* poss, const int32_t* n_sels,
                                     void* const* k_outs, void* const* v_outs, cudaStream_t s);

cudaError_t launch_timeout_probe(rkv_ctx* c, cudaStream_t s);

// Sparse attention over restored K/V: at most kAttnMaxChunks chunks of selected tokens
// (of attention_chunk(n) tokens each), query heads per key/value head <= kAttnMaxGroup.
constexpr int kAttnMaxChunks = 256;
constexpr int kAttnMaxGroup = 8;
constexpr int kAttnMaxTokens = kAttnMaxChunks * 1024;
int attention_chunk(int n, int N, int num_sms);
cudaError_t launch_attention(rkv_ctx* c, const float* q, int n_q_heads, const void* k,
                             const void* v, int n, float* out, cudaStream_t s);

// Restore fused into the sparse attention (D = 128, bf16 K_hat / V_hat, n_q_heads / N <=
// kAttnMaxGroup, n_sel <= kAttnMaxTokens): per (token tile, query head) softmax partials
// in the context's workspace, then launch_attend_merge.
cudaError_t launch_restore_attend(rkv_ctx* c, const int32_t* seq, const int32_t* pos, int n_sel,
                                  const float* q, int n_q_heads, float* out, cudaStream_t s);
// out[h] = sum_t o_t[h] e^(m_t[h] - M) / sum_t l_t[h] e^(m_t[h] - M), M = max_t m_t[h], over
// `tiles` partials [tiles][n_q_heads] (o: [tiles][n_q_heads][128]).
cudaError_t launch_attend_merge(rkv_ctx* c, const float* pm, const float* pl, const float* po,
                                int tiles, int n_q_heads, float* out, cudaStream_t s);

// Record the message rkv_last_error returns on this thread.
void set_error(const char* msg);

// Instrumentation helpers used around every launch.
void timing_begin(rkv_ctx* c, const char* name, cudaStream_t s, cudaEvent_t* start);
void timing_end(rkv_ctx* c, const char* name, cudaStream_t s, cudaEvent_t start);

}  // namespace rkv
