// Shared device helpers of libnt: dtype traits, vector loads/stores, the
// device status word and the internal launcher declarations.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/nt.h"

namespace nt {

// Bits of the device status word (see nt_device_status).
enum : unsigned int {
  kDevTimeout = 1u,      // a bounded wait ran out
  kDevCheck = 2u,        // a data check failed
};

typedef __nv_bfloat16 bf16;

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// Number of SMs of the current device (cached per device).
int sm_count();

// Records a one-line detail for nt_last_error() and returns `s`.
nt_status record_error(nt_status s, const char* msg);

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// Load 8 consecutive elements (16 bytes of bf16, 32 bytes of fp32) as fp32.
__device__ __forceinline__ void load8(const bf16* p, float* out) {
  uint4 raw = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    out[2 * i] = f.x;
    out[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float* out) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
  out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
}
__device__ __forceinline__ void store8(bf16* p, const float* in) {
  uint4 raw;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = raw;
}
__device__ __forceinline__ void store8(float* p, const float* in) {
  *reinterpret_cast<float4*>(p) = make_float4(in[0], in[1], in[2], in[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(in[4], in[5], in[6], in[7]);
}
// Streaming store (evict-first): output that is not read again soon.
__device__ __forceinline__ void store8_stream(bf16* p, const float* in) {
  uint4 raw;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
  __stcs(reinterpret_cast<uint4*>(p), raw);
}
__device__ __forceinline__ void store8_stream(float* p, const float* in) {
  __stcs(reinterpret_cast<float4*>(p), make_float4(in[0], in[1], in[2], in[3]));
  __stcs(reinterpret_cast<float4*>(p + 4), make_float4(in[4], in[5], in[6], in[7]));
}

__device__ __forceinline__ void flag_device(unsigned int* status, unsigned int bits) {
  if (status) atomicOr(status, bits);
}

// Programmatic dependent launch.  A kernel started by launch_pdl may begin
// while the kernel before it in the stream is still running: every thread
// calls pdl_wait() before it reads or writes global memory that kernel
// touches (the wait returns once that kernel has completed and its writes
// are visible).  pdl_trigger() lets the next kernel in the stream start its
// CTAs early.  Both are no-ops in a kernel launched the ordinary way.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ----------------------------------------------------------------------------
// Internal launchers (one per kernel family), called by the ABI layer after
// argument validation.  Each returns cudaGetLastError() of its launches.
// ----------------------------------------------------------------------------
// Column side of a partition (rectangular pair states); square partitions
// may leave col_lengths NULL, which means M_i = N_i.
inline const int32_t* col_lengths_of(const nt_partition* p) { return p->col_lengths ? p->col_lengths : p->lengths; }
inline const int32_t* col_cu_of(const nt_partition* p) {
  return p->col_lengths ? p->col_cu_seqlens : p->cu_seqlens;
}
inline int64_t t_cols_of(const nt_partition* p) { return p->col_lengths ? p->T_cols : p->T; }
inline int32_t max_cols_of(const nt_partition* p) { return p->col_lengths ? p->max_col_len : p->max_len; }

// cols / cu_cols NULL: square (M_i = N_i).  totals = {T, P, max_len, check,
// T_cols, max_col_len} (the last two only with cols).  host_totals (nullable):
// a device-accessible alias of mapped pinned host memory that receives the
// same totals, so the host reads them after a stream sync with no copy.
cudaError_t launch_partition_scan(const int32_t* lengths, const int32_t* cols, int32_t B, int32_t* cu,
                                  int32_t* cu_cols, int64_t* pair_off, int64_t* totals, int64_t* host_totals,
                                  cudaStream_t s);
cudaError_t launch_partition_rows(const int32_t* lengths, const int32_t* cols, const int32_t* cu,
                                  const int64_t* pair_off, int32_t B, int64_t T, int64_t P, int64_t* row_start,
                                  int32_t* row_sample, cudaStream_t s);
// Row splits after the scan in the same stream, T and P from the device
// totals, writes bounded by the capacity cap (rows of row_start: cap + 1).
cudaError_t launch_partition_rows_dev(const int32_t* lengths, const int32_t* cols, const int32_t* cu,
                                      const int64_t* pair_off, int32_t B, const int64_t* totals, int64_t cap,
                                      int64_t* row_start, int32_t* row_sample, cudaStream_t s);
// Square partitions of small batches (partition_fused_fits): the scan and the
// row splits of the two calls above in one single-CTA launch, same outputs.
bool partition_fused_fits(int32_t B, int64_t cap);
cudaError_t launch_partition_fused(const int32_t* lengths, int32_t B, int64_t cap, int32_t* cu, int64_t* pair_off,
                                   int64_t* totals, int64_t* row_start, int32_t* row_sample, int64_t* host_totals,
                                   cudaStream_t s);

// Y[M, N] = X[M, K] W[N, K]^T (+ bias[N]) (+ R[M, N]).  Up to two independent
// problems in one launch (gridDim.z); all row-major, contiguous.
struct LinearProblem {
  const void* X; const void* W; const float* bias; const void* R; void* Y;   // Y = X W^T (+ bias) (+ R)
};
cudaError_t launch_linear(int in_dtype /*nt_dtype of X, W, R*/, int out_f32 /*Y fp32?*/,
                          const LinearProblem* probs, int nprob, int64_t M, int N, int K,
                          cudaStream_t s);

// Same problem on the tcgen05 tensor cores: bf16 X and W, N % 128 == 0,
// K % 64 == 0; Y fp32 (out_f32) or bf16.
bool linear_tc_supported(int in_dtype, int64_t M, int N, int K);
cudaError_t launch_linear_tc(int out_f32, const LinearProblem* probs, int nprob, int64_t M, int N, int K,
                             unsigned int* status, cudaStream_t s);
// Two problems on one output tile grid, as the block backward needs them:
// Y = ReLU(X W^T + bias) and Y2 = (X2 W2^T) where bf16(Y) > 0 (X [M, K],
// W [N, K], X2 [M, K2], W2 [N, K2], Y and Y2 [M, N], all bf16 row-major;
// N % 128 == 0, K and K2 multiples of 64).  Persistent CTAs.
cudaError_t launch_linear_tc_dual(const void* X, const void* W, const float* bias, const void* X2, const void* W2,
                                  void* Y, void* Y2, int64_t M, int N, int K, int K2, unsigned int* status,
                                  cudaStream_t s);

cudaError_t launch_broadcast(nt_dtype dt, const float* u, const float* v, const nt_partition* p,
                             int C_z, void* z, cudaStream_t s);

// W3 == NULL: ReLU update; W3 given: SwiGLU update SiLU(W1 x + b1) * (W3 x + b3).
cudaError_t launch_transition_simt(nt_dtype dt, const void* z_in, void* z_out, int64_t P, int C_z,
                                   int H_t, const float* gamma, const float* beta, float eps,
                                   const void* W1, const float* b1, const void* W3, const float* b3,
                                   const void* W2, const float* b2, cudaStream_t s);
bool transition_tc_supported(nt_dtype dt, int C_z, int H_t, bool glu);
cudaError_t launch_transition_tc(const void* z_in, void* z_out, int64_t P, int C_z, int H_t,
                                 const float* gamma, const float* beta, float eps, const void* W1,
                                 const float* b1, const void* W3, const float* b3, const void* W2,
                                 const float* b2, unsigned int* status, cudaStream_t s);

// The column mean; with sq_part (C_z a multiple of 8, reduce_sq_supported),
// also Eq. 5's weighted pair squares, one double per CTA into sq_part, their
// count into *sq_parts (at most kReduceMaxGrid).
constexpr int64_t kReduceMaxGrid = 8192;
bool reduce_sq_supported(int C_z);
cudaError_t launch_reduce(nt_dtype dt, const void* z, const nt_partition* p, int C_z, void* m, cudaStream_t s,
                          double* sq_part = nullptr, int* sq_parts = nullptr);
// Fused block: the transition kernel building z from u, v and summing rows
// into m_acc (fp32, zeroed by the caller); then m = m_acc / M_i.
cudaError_t launch_block_fused_tc(const float* u, const float* v, const nt_partition* part, void* z_out, int C_z,
                                  int H_t, const float* gamma, const float* beta, float eps, const void* W1,
                                  const float* b1, const void* W3, const float* b3, const void* W2, const float* b2,
                                  float* m_acc, unsigned int* status, cudaStream_t s);
cudaError_t launch_mean_finish(nt_dtype dt, const float* m_acc, const nt_partition* p, int C_z, void* m,
                               cudaStream_t s);

// One varlen attention problem: queries [cu_q[b], cu_q[b+1]) attend to keys
// [cu_k[b], cu_k[b+1]) (cu_k == cu_q for self-attention); causal masks key j
// of a segment for query i when j > i + (n_k - n_q).
struct AttnProblem {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* cu_q;
  const int32_t* cu_k;
  int32_t B;
  int64_t T_q, T_k;
  int32_t max_len_q;
  int H, d;
  float scale;
  bool causal;
  void* o;
  float* lse;
  // Caller-owned work counter of the persistent schedule (one 32-bit word,
  // cleared on the launch's stream), or NULL: one CTA per work item then.
  unsigned int* work;
};

// Backward of one varlen attention problem (the forward's q, k, v, o, its
// natural-log lse, and the upstream gradient d_o; outputs dq, dk, dv).
struct AttnBwdProblem {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* d_o;
  const float* lse;
  const int32_t* cu_q;
  const int32_t* cu_k;
  int32_t B;
  int64_t T_q, T_k;
  int32_t max_len_q, max_len_k;
  int H, d;
  float scale;
  bool causal;
  void* dq;
  void* dk;
  void* dv;
  // Caller-owned work counters of the persistent dK/dV and dQ kernels (two
  // 32-bit words, cleared on the launch's stream), or NULL: one CTA per
  // work item then.
  unsigned int* work;
};
bool attn_bwd_supported(int d);
// Dbuf: H * T_q fp32 of device workspace (rowsum(dO * O)).
cudaError_t launch_attn_bwd(nt_dtype dt, const AttnBwdProblem& p, float* Dbuf, unsigned int* status, cudaStream_t s);
// The tensor-core kernels (dK/dV, then dQ) after Dbuf holds rowsum(dO * O);
// T_q, T_k and B must be > 0.
bool attn_bwd_tc_supported(nt_dtype dt, int d);
cudaError_t launch_attn_bwd_tc(const AttnBwdProblem& p, float* Dbuf, unsigned int* status, cudaStream_t s);

// The Eq. 5 loss ("DanLing NestedTensor" Appendix A.1) on the block's outputs
// and, optionally, its gradients dX~ [T, C_s] and dP~ [P, C_z] (fp32).
// workspace: eq5_loss_workspace_bytes() for the partial sums.
size_t eq5_loss_workspace_bytes();
// The loss with its pair term already summed by the reduce (pair_sq: npair
// weighted partials): the single-row term here, then one fixed-order finish.
cudaError_t launch_eq5_loss_rows(nt_dtype dt, const nt_partition* p, const void* s_out, int C_s, int C_z,
                                 float* loss, const double* pair_sq, int npair, void* workspace, cudaStream_t s);
cudaError_t launch_eq5_loss(nt_dtype dt, const nt_partition* p, const void* s_out, int C_s, const void* z_tilde,
                            int C_z, float* loss, float* ds_out, float* dz, void* workspace, cudaStream_t s);

// The block's backward (the chain rule of Eq. 1) for upstream gradients
// ds_out [T, C_s] and dz_up [P, C_z] (nullable), fp32; square partitions.
// u, v, dM, dz, du, dv are fp32 scratch the caller provides ([T, C_z] each,
// dz [P, C_z]); u and v must hold s W_a^T, s W_b^T.  The gradient outputs
// that are sums (every weight and bias gradient) must be zero on entry.
struct BlockBwd {
  const nt_partition* part;
  int C_s, C_z, H_t;
  const void* s;
  const void* W_a;
  const void* W_b;
  const float* gamma;
  const float* beta;
  float eps;
  const void* W1;
  const float* b1;
  const void* W2;
  const void* W_g;
  const void* m;
  const float* ds_out;
  const float* dz_up;
  // the tensor-core route only: when set, the upstream pair gradient is
  // Eq. 5's, gp_b z~ (z~ [P, C_z] bf16), formed where it is read; dz_up is
  // then unused
  const void* zt_up;
  float* ds;
  float* dW_a;
  float* dW_b;
  float* dgamma;
  float* dbeta;
  float* dW1;
  float* db1;
  float* dW2;
  float* db2;
  float* dW_g;
  float* db_g;
  float* u;
  float* v;
  float* dM;
  float* dz;
  float* du;
  float* dv;
  // the tensor-core route's buffers (bf16, C_z = 128, H_t % 128 == 0), else null
  void* tc_ws;
};
bool block_bwd_supported(int C_z, int H_t);
// Whether the pair-cell part runs on the tensor cores, and the workspace the
// backward needs: (5 T + P) C_z fp32 words, plus the route's cell rows.
bool block_bwd_tc(nt_dtype dt, int64_t P, int C_z, int H_t);
size_t block_bwd_workspace_bytes(nt_dtype dt, int64_t T, int64_t P, int C_z, int H_t);
cudaError_t launch_block_backward(nt_dtype dt, const BlockBwd& q, unsigned int* status, cudaStream_t s);

// Weight gradients over the cells on the tensor cores: G[M, N] = A^T B and
// optionally colsum[M] = sum of A's rows, A [P, M] and B [P, N] bf16
// row-major with rows lda and ldb elements apart (multiples of 8), G and
// colsum fp32 (written, not added to); M, N multiples of 128.
bool wgrad_tc_supported(int64_t P, int M, int N);
size_t wgrad_tc_workspace_bytes(int64_t P, int M, int N);
cudaError_t launch_wgrad_tc(const void* A, int lda, const void* B, int ldb, int64_t P, int M, int N, float* G,
                            float* colsum, void* workspace, unsigned int* status, cudaStream_t s);

bool attn_simt_supported(int d);
cudaError_t launch_attn_simt(nt_dtype dt, const AttnProblem& p, unsigned int* status, cudaStream_t s);
bool attn_tc_supported(nt_dtype dt, int d);
cudaError_t launch_attn_tc(const AttnProblem& p, unsigned int* status, cudaStream_t s);
cudaError_t launch_selftest_wait(int mode, uint64_t delay_ns, uint64_t limit_ns, int64_t* result,
                                 unsigned int* status, cudaStream_t s);

}  // namespace nt
