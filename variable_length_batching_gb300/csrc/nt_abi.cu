// The C ABI of libnt (declared in include/nt.h): argument validation on the
// host, then one batch-level launch per step on the caller's stream -- every
// call covers the whole packed batch, never one call per sample ("DanLing
// NestedTensor" section 4.4, "Separating interface cost from execution
// strategy": segmented calls over the batch).
#include <cstdarg>
#include <cstdio>
#include <cmath>
#include <cstring>
#include <mutex>

#include "nt_common.cuh"

namespace nt {

// Device status word: set by device-side checks, read by nt_device_status.
__device__ unsigned int g_device_status;

namespace {

thread_local char g_last_error[512] = "";

nt_status fail(nt_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

nt_status cuda_fail(cudaError_t e, const char* where) {
  return fail(NT_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxDevices = 64;
std::mutex g_status_mu;
unsigned int* g_status_ptr[kMaxDevices] = {};

// Device address of g_device_status on the current device, looked up once
// per device with that device current.
unsigned int* status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned int*>(p);
  }
  return g_status_ptr[dev];
}

constexpr uint64_t kSelftestMaxNs = 2000000000ull;   // the longest wait or delay of the self-test
constexpr int64_t kMaxCells = 0x7fffffffLL - 1024;     // pair cells a transition or fused call takes

bool width_ok(nt_dtype dt, int64_t w) { return w > 0 && w % (dt == NT_BF16 ? 8 : 4) == 0; }
bool dtype_ok(nt_dtype dt) { return dt == NT_F32 || dt == NT_BF16; }
size_t esize(nt_dtype dt) { return dt == NT_BF16 ? 2 : 4; }

nt_status check_partition(const nt_partition* p, bool need_rows) {
  if (!p) return fail(NT_ERR_INVALID, "partition is NULL");
  if (p->B < 0 || p->T < 0 || p->P < 0 || p->max_len < 0)
    return fail(NT_ERR_INVALID, "partition has negative sizes");
  if (p->T > 0 && (!p->lengths || !p->cu_seqlens || !p->pair_off))
    return fail(NT_ERR_INVALID, "partition pointers are NULL");
  if (need_rows && p->T > 0 && (!p->row_start || !p->row_sample))
    return fail(NT_ERR_INVALID, "partition has no row splits (call nt_partition_rows)");
  if (p->col_lengths) {
    if (p->T_cols < 0 || p->max_col_len < 0 || (p->T_cols > 0 && !p->col_cu_seqlens))
      return fail(NT_ERR_INVALID, "partition column fields are inconsistent");
    if (p->T > 0 && p->P > p->T * (int64_t)p->max_col_len)
      return fail(NT_ERR_INVALID, "partition totals are inconsistent (T=%lld P=%lld max_col_len=%d)",
                  (long long)p->T, (long long)p->P, p->max_col_len);
  } else if (p->P < p->T || (p->T > 0 && p->P > p->T * (int64_t)p->max_len)) {
    return fail(NT_ERR_INVALID, "partition totals are inconsistent (T=%lld P=%lld max_len=%d)",
                (long long)p->T, (long long)p->P, p->max_len);
  }
  return NT_OK;
}

}  // namespace

nt_status record_error(nt_status s, const char* msg) { return fail(s, "%s", msg); }

int sm_count() {
  static int cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace nt

using namespace nt;

namespace {

// Device workspace of the attention calls' persistent schedules: their work
// counters (a few 32-bit words), padded to 256 bytes.
constexpr size_t kAttnWorkBytes = 256;

// Byte offset of the backward's two work counters in its workspace, after
// the H * T_q fp32 row sums rowsum(dO * O) (256-byte aligned).
size_t bwd_counter_offset(int64_t T_q, int32_t H) {
  return ((size_t)T_q * (size_t)H * sizeof(float) + 255) & ~(size_t)255;
}

// The residual transition of P cells with the ReLU update (W3 == NULL) or
// the SwiGLU one.
nt_status transition_cells(int64_t P, nt_dtype dtype, const void* z_in, void* z_out, int32_t C_z, int32_t H_t,
                           const float* ln_gamma, const float* ln_beta, float ln_eps, const void* W1,
                           const float* b1, const void* W3, const float* b3, const void* W2, const float* b2,
                           void* stream) {
  if (P < 0) return fail(NT_ERR_INVALID, "cell count %lld < 0", (long long)P);
  if (!dtype_ok(dtype)) return fail(NT_ERR_INVALID, "bad dtype %d", (int)dtype);
  if (P == 0) return NT_OK;                  // nothing to map (the pointers of empty tensors may be NULL)
  // cell rows are 32-bit TMA coordinates (2^31 bf16 cells of 128 features
  // would be 550 GB, beyond the device anyway)
  if (P > kMaxCells) return fail(NT_ERR_OVERFLOW, "%lld cells: at most %lld", (long long)P, (long long)kMaxCells);
  if (!width_ok(dtype, C_z) || !width_ok(dtype, H_t))
    return fail(NT_ERR_UNSUPPORTED, "C_z=%d, H_t=%d must be positive multiples of %d", C_z, H_t,
                dtype == NT_BF16 ? 8 : 4);
  if (!z_in || !z_out || !ln_gamma || !ln_beta || !W1 || !W2)
    return fail(NT_ERR_INVALID, "NULL pointer");
  if (!aligned16(z_in) || !aligned16(z_out) || !aligned16(W1) || !aligned16(W2) || !aligned16(W3) ||
      !aligned16(ln_gamma) || !aligned16(ln_beta) || !aligned16(b1) || !aligned16(b2) || !aligned16(b3))
    return fail(NT_ERR_INVALID, "pointers must be 16-byte aligned");
  if (!(ln_eps >= 0.0f)) return fail(NT_ERR_INVALID, "ln_eps must be >= 0");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (transition_tc_supported(dtype, C_z, H_t, W3 != nullptr)) {
    e = launch_transition_tc(z_in, z_out, P, C_z, H_t, ln_gamma, ln_beta, ln_eps, W1, b1, W3, b3, W2,
                             b2, status_word(), s);
    if (e != cudaSuccess) return cuda_fail(e, "transition (tensor core) launch");
    return NT_OK;
  }
  if (sizeof(float) * 8 * (size_t)(C_z + H_t) > 200 * 1024)
    return fail(NT_ERR_UNSUPPORTED, "C_z + H_t = %d too wide for the CUDA-core transition", C_z + H_t);
  e = launch_transition_simt(dtype, z_in, z_out, P, C_z, H_t, ln_gamma, ln_beta, ln_eps, W1,
                             b1, W3, b3, W2, b2, s);
  if (e != cudaSuccess) return cuda_fail(e, "transition launch");
  return NT_OK;
}

nt_status pair_transition(const nt_partition* part, nt_dtype dtype, const void* z_in, void* z_out, int32_t C_z,
                          int32_t H_t, const float* ln_gamma, const float* ln_beta, float ln_eps, const void* W1,
                          const float* b1, const void* W3, const float* b3, const void* W2, const float* b2,
                          void* stream) {
  nt_status st = check_partition(part, false);
  if (st != NT_OK) return st;
  return transition_cells(part->P, dtype, z_in, z_out, C_z, H_t, ln_gamma, ln_beta, ln_eps, W1, b1, W3, b3, W2,
                          b2, stream);
}

// u = s_left W_a^T (T rows), v = s_right W_b^T (T_cols rows), fp32.
cudaError_t project_uv(const nt_partition* part, nt_dtype dtype, const void* s_left, const void* s_right,
                       int32_t C_s, const void* W_a, const void* W_b, int32_t C_z, float* u, float* v,
                       cudaStream_t s) {
  const int64_t T_cols = t_cols_of(part);
  LinearProblem probs[2] = {{s_left, W_a, nullptr, nullptr, u}, {s_right, W_b, nullptr, nullptr, v}};
  if (T_cols == part->T)   // one launch for both projections
    return linear_tc_supported(dtype, part->T, C_z, C_s)
               ? launch_linear_tc(1, probs, 2, part->T, C_z, C_s, status_word(), s)
               : launch_linear(dtype, 1, probs, 2, part->T, C_z, C_s, s);
  // rectangular: row and column singles have different row counts
  const int64_t rows[2] = {part->T, T_cols};
  cudaError_t e = cudaSuccess;
  for (int k = 0; k < 2 && e == cudaSuccess; ++k) {
    if (rows[k] == 0) continue;
    e = linear_tc_supported(dtype, rows[k], C_z, C_s)
            ? launch_linear_tc(1, &probs[k], 1, rows[k], C_z, C_s, status_word(), s)
            : launch_linear(dtype, 1, &probs[k], 1, rows[k], C_z, C_s, s);
  }
  return e;
}

// The checks of the backward's arguments that do not depend on how its
// upstream gradients arrive.
nt_status check_block_backward(const nt_partition* part, nt_dtype dtype, int32_t C_s, int32_t C_z, int32_t H_t,
                               float ln_eps) {
  nt_status st = check_partition(part, true);
  if (st != NT_OK) return st;
  if (part->col_lengths && (part->col_lengths != part->lengths || part->col_cu_seqlens != part->cu_seqlens))
    return fail(NT_ERR_UNSUPPORTED, "the block backward takes square partitions");
  if (!dtype_ok(dtype)) return fail(NT_ERR_INVALID, "bad dtype %d", (int)dtype);
  if (!width_ok(dtype, C_s) || !width_ok(dtype, C_z) || !block_bwd_supported(C_z, H_t))
    return fail(NT_ERR_UNSUPPORTED, "C_s=%d, C_z=%d (8..128), H_t=%d (a multiple of 64)", C_s, C_z, H_t);
  if (!(ln_eps >= 0.0f)) return fail(NT_ERR_INVALID, "ln_eps must be >= 0");
  return NT_OK;
}

// The backward proper (arguments checked): zt_up non-NULL only on the
// tensor-core route, for Eq. 5's upstream pair gradient formed from z~.
nt_status block_backward_run(const nt_partition* part, nt_dtype dtype, const void* s, int32_t C_s, const void* W_a,
                             const void* W_b, int32_t C_z, int32_t H_t, const float* ln_gamma, const float* ln_beta,
                             float ln_eps, const void* W1, const float* b1, const void* W2, const void* W_g,
                             const void* m, const float* ds_out, const float* dz_tilde, const void* zt_up, float* ds,
                             float* dW_a, float* dW_b, float* dgamma, float* dbeta, float* dW1, float* db1,
                             float* dW2, float* db2, float* dW_g, float* db_g, void* workspace, cudaStream_t st_) {
  // the gradients that are sums start at zero
  const size_t f4 = sizeof(float);
  struct { float* p; size_t n; } zero[] = {
      {dW_a, (size_t)C_z * C_s}, {dW_b, (size_t)C_z * C_s}, {dgamma, (size_t)C_z}, {dbeta, (size_t)C_z},
      {dW1, (size_t)H_t * C_z}, {db1, (size_t)H_t}, {dW2, (size_t)C_z * H_t}, {db2, (size_t)C_z},
      {dW_g, (size_t)C_s * C_z}, {db_g, (size_t)C_s}};
  for (auto& zr : zero) {
    cudaError_t e = cudaMemsetAsync(zr.p, 0, zr.n * f4, st_);
    if (e != cudaSuccess) return cuda_fail(e, "gradient clear");
  }
  if (part->T == 0) return NT_OK;
  float* u = static_cast<float*>(workspace);
  float* v = u + part->T * (int64_t)C_z;
  float* dM = v + part->T * (int64_t)C_z;
  float* du = dM + part->T * (int64_t)C_z;
  float* dv = du + part->T * (int64_t)C_z;
  float* dz = dv + part->T * (int64_t)C_z;
  cudaError_t e = project_uv(part, dtype, s, s, C_s, W_a, W_b, C_z, u, v, st_);
  if (e != cudaSuccess) return cuda_fail(e, "projection launch");
  // the tensor-core route's buffers follow the CUDA-core route's
  const size_t base = ((size_t)(5 * part->T + part->P) * (size_t)C_z * sizeof(float) + 255) & ~(size_t)255;
  void* tc_ws = block_bwd_tc(dtype, part->P, C_z, H_t) ? static_cast<uint8_t*>(workspace) + base : nullptr;
  BlockBwd q = {part, C_s, C_z, H_t, s, W_a, W_b, ln_gamma, ln_beta, ln_eps, W1, b1, W2, W_g, m, ds_out, dz_tilde,
                zt_up, ds, dW_a, dW_b, dgamma, dbeta, dW1, db1, dW2, db2, dW_g, db_g, u, v, dM, dz, du, dv, tc_ws};
  unsigned int* status = status_word();
  if (!status) return fail(NT_ERR_CUDA, "device status word unavailable");
  e = launch_block_backward(dtype, q, status, st_);
  if (e != cudaSuccess) return cuda_fail(e, "block backward launch");
  return NT_OK;
}

// Workspace of the fused loss + backward: the loss's partial sums, dX~
// ([T, C_s] fp32), on routes other than the tensor-core one dL/dz~ ([P, C_z]
// fp32), then the backward's own (each part 256-byte aligned).
struct LossBwdLayout {
  size_t dx, dz, bwd, end;
};
LossBwdLayout loss_bwd_layout(nt_dtype dtype, int64_t T, int64_t P, int32_t C_s, int32_t C_z, int32_t H_t) {
  auto a256 = [](size_t x) { return (x + 255) & ~(size_t)255; };
  LossBwdLayout L;
  L.dx = a256(eq5_loss_workspace_bytes());
  L.dz = a256(L.dx + (size_t)T * C_s * sizeof(float));
  const size_t dz_bytes = block_bwd_tc(dtype, P, C_z, H_t) ? 0 : (size_t)P * C_z * sizeof(float);
  L.bwd = a256(L.dz + dz_bytes);
  L.end = L.bwd + block_bwd_workspace_bytes(dtype, T, P, C_z, H_t);
  return L;
}

}  // namespace

extern "C" {

const char* nt_status_str(nt_status s) {
  switch (s) {
    case NT_OK: return "NT_OK";
    case NT_ERR_INVALID: return "NT_ERR_INVALID";
    case NT_ERR_UNSUPPORTED: return "NT_ERR_UNSUPPORTED";
    case NT_ERR_OVERFLOW: return "NT_ERR_OVERFLOW";
    case NT_ERR_CUDA: return "NT_ERR_CUDA";
    case NT_ERR_TIMEOUT: return "NT_ERR_TIMEOUT";
    case NT_ERR_DEVICE_CHECK: return "NT_ERR_DEVICE_CHECK";
  }
  return "NT_ERR_UNKNOWN";
}

const char* nt_last_error(void) { return g_last_error; }

// The partition's totals come back through a small mapped pinned buffer per
// host thread (allocated on first use, kept for the process).  The scan
// kernel writes them there itself, through the buffer's device alias, so the
// host needs only a stream sync and no copy engine: a copy would queue
// behind any large device-to-host transfer in flight on another stream.  If
// mapping fails, the totals are copied back (to pageable memory if pinning
// fails too).
struct PinnedTotals {
  int64_t* host = nullptr;
  int64_t* dev = nullptr;     // device alias of host; null when not mapped
  bool tried = false;
};

static PinnedTotals& pinned_totals() {
  static thread_local PinnedTotals p;
  if (!p.tried) {
    p.tried = true;
    void* h = nullptr;
    if (cudaHostAlloc(&h, 8 * sizeof(int64_t), cudaHostAllocMapped | cudaHostAllocPortable) == cudaSuccess) {
      p.host = static_cast<int64_t*>(h);
      void* d = nullptr;
      if (cudaHostGetDevicePointer(&d, h, 0) == cudaSuccess) p.dev = static_cast<int64_t*>(d);
    }
    cudaGetLastError();
  }
  return p;
}

// `mapped`: the launch was given pinned_totals().dev, so the totals are
// already on their way to the host buffer.
static cudaError_t read_totals(int64_t* host, const int64_t* d_totals, int n, cudaStream_t s, bool mapped) {
  PinnedTotals& p = pinned_totals();
  cudaError_t e;
  if (mapped) {
    e = cudaStreamSynchronize(s);
    if (e == cudaSuccess)
      for (int i = 0; i < n; ++i) host[i] = reinterpret_cast<volatile int64_t*>(p.host)[i];
    return e;
  }
  int64_t* dst = p.host ? p.host : host;
  e = cudaMemcpyAsync(dst, d_totals, n * sizeof(int64_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && p.host)
    for (int i = 0; i < n; ++i) host[i] = p.host[i];
  return e;
}

nt_status nt_partition_build(const int32_t* d_lengths, int32_t B, int32_t* d_cu_seqlens,
                             int64_t* d_pair_off, int64_t* d_totals, nt_partition* out,
                             void* stream) {
  if (!out) return fail(NT_ERR_INVALID, "out is NULL");
  if (B < 0) return fail(NT_ERR_INVALID, "B = %d < 0", B);
  if ((B > 0 && !d_lengths) || !d_cu_seqlens || !d_pair_off || !d_totals)
    return fail(NT_ERR_INVALID, "NULL device pointer");
  if (!aligned16(d_totals) || !aligned16(d_pair_off) || !aligned16(d_cu_seqlens))
    return fail(NT_ERR_INVALID, "pointers must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int64_t* ht = pinned_totals().dev;
  cudaError_t e = launch_partition_scan(d_lengths, nullptr, B, d_cu_seqlens, nullptr, d_pair_off, d_totals, ht, s);
  if (e != cudaSuccess) return cuda_fail(e, "partition scan launch");
  int64_t tot[4] = {0, 0, 0, 0};
  e = read_totals(tot, d_totals, 4, s, ht != nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "partition totals readback");
  out->B = B;
  out->T = tot[0];
  out->P = tot[1];
  out->max_len = (int32_t)tot[2];
  out->lengths = d_lengths;
  out->cu_seqlens = d_cu_seqlens;
  out->pair_off = d_pair_off;
  out->row_start = nullptr;
  out->row_sample = nullptr;
  // square: the column side is the row side
  out->col_lengths = d_lengths;
  out->col_cu_seqlens = d_cu_seqlens;
  out->T_cols = tot[0];
  out->max_col_len = (int32_t)tot[2];
  if (tot[3] & 1) return fail(NT_ERR_INVALID, "a sample length is negative");
  if (tot[3] & 2) return fail(NT_ERR_OVERFLOW, "T = %lld does not fit int32 cu_seqlens", (long long)tot[0]);
  return NT_OK;
}

nt_status nt_partition_build_rect(const int32_t* d_rows, const int32_t* d_cols, int32_t B,
                                  int32_t* d_cu_rows, int32_t* d_cu_cols, int64_t* d_pair_off,
                                  int64_t* d_totals, nt_partition* out, void* stream) {
  if (!out) return fail(NT_ERR_INVALID, "out is NULL");
  if (B < 0) return fail(NT_ERR_INVALID, "B = %d < 0", B);
  if ((B > 0 && (!d_rows || !d_cols)) || !d_cu_rows || !d_cu_cols || !d_pair_off || !d_totals)
    return fail(NT_ERR_INVALID, "NULL device pointer");
  if (!aligned16(d_totals) || !aligned16(d_pair_off) || !aligned16(d_cu_rows) || !aligned16(d_cu_cols))
    return fail(NT_ERR_INVALID, "pointers must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int64_t* ht = pinned_totals().dev;
  cudaError_t e = launch_partition_scan(d_rows, B > 0 ? d_cols : d_rows, B, d_cu_rows, d_cu_cols, d_pair_off,
                                        d_totals, ht, s);
  if (e != cudaSuccess) return cuda_fail(e, "partition scan launch");
  int64_t tot[6] = {0, 0, 0, 0, 0, 0};
  e = read_totals(tot, d_totals, 6, s, ht != nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "partition totals readback");
  out->B = B;
  out->T = tot[0];
  out->P = tot[1];
  out->max_len = (int32_t)tot[2];
  out->lengths = d_rows;
  out->cu_seqlens = d_cu_rows;
  out->pair_off = d_pair_off;
  out->row_start = nullptr;
  out->row_sample = nullptr;
  out->col_lengths = B > 0 ? d_cols : d_rows;
  out->col_cu_seqlens = d_cu_cols;
  out->T_cols = B > 0 ? tot[4] : 0;
  out->max_col_len = B > 0 ? (int32_t)tot[5] : 0;
  if (tot[3] & 1) return fail(NT_ERR_INVALID, "a sample length is negative");
  if (tot[3] & 2) return fail(NT_ERR_OVERFLOW, "sum N_i = %lld does not fit int32", (long long)tot[0]);
  if (tot[3] & 4) return fail(NT_ERR_OVERFLOW, "sum M_i = %lld does not fit int32", (long long)tot[4]);
  return NT_OK;
}

nt_status nt_partition_build_with_rows(const int32_t* d_lengths, int32_t B, int64_t T_cap, int32_t* d_cu_seqlens,
                                       int64_t* d_pair_off, int64_t* d_totals, int64_t* d_row_start,
                                       int32_t* d_row_sample, nt_partition* out, void* stream) {
  if (!out) return fail(NT_ERR_INVALID, "out is NULL");
  if (B < 0) return fail(NT_ERR_INVALID, "B = %d < 0", B);
  if (T_cap < 0) return fail(NT_ERR_INVALID, "T_cap = %lld < 0", (long long)T_cap);
  if ((B > 0 && !d_lengths) || !d_cu_seqlens || !d_pair_off || !d_totals || !d_row_start ||
      (T_cap > 0 && !d_row_sample))
    return fail(NT_ERR_INVALID, "NULL device pointer");
  if (!aligned16(d_totals) || !aligned16(d_pair_off) || !aligned16(d_cu_seqlens) || !aligned16(d_row_start) ||
      !aligned16(d_row_sample))
    return fail(NT_ERR_INVALID, "pointers must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int64_t* ht = pinned_totals().dev;
  cudaError_t e;
  if (partition_fused_fits(B, T_cap)) {
    e = launch_partition_fused(d_lengths, B, T_cap, d_cu_seqlens, d_pair_off, d_totals, d_row_start, d_row_sample,
                               ht, s);
  } else {
    e = launch_partition_scan(d_lengths, nullptr, B, d_cu_seqlens, nullptr, d_pair_off, d_totals, ht, s);
    if (e == cudaSuccess)
      e = launch_partition_rows_dev(d_lengths, nullptr, d_cu_seqlens, d_pair_off, B, d_totals, T_cap, d_row_start,
                                    d_row_sample, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "partition launch");
  int64_t tot[4] = {0, 0, 0, 0};
  e = read_totals(tot, d_totals, 4, s, ht != nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "partition totals readback");
  out->B = B;
  out->T = tot[0];
  out->P = tot[1];
  out->max_len = (int32_t)tot[2];
  out->lengths = d_lengths;
  out->cu_seqlens = d_cu_seqlens;
  out->pair_off = d_pair_off;
  out->row_start = d_row_start;
  out->row_sample = d_row_sample;
  out->col_lengths = d_lengths;
  out->col_cu_seqlens = d_cu_seqlens;
  out->T_cols = tot[0];
  out->max_col_len = (int32_t)tot[2];
  if (tot[3] & 1) return fail(NT_ERR_INVALID, "a sample length is negative");
  if (tot[3] & 2) return fail(NT_ERR_OVERFLOW, "T = %lld does not fit int32 cu_seqlens", (long long)tot[0]);
  if (tot[0] > T_cap)
    return fail(NT_ERR_INVALID, "the lengths sum to T = %lld > T_cap = %lld: row splits incomplete",
                (long long)tot[0], (long long)T_cap);
  return NT_OK;
}

nt_status nt_partition_rows(nt_partition* part, int64_t* d_row_start, int32_t* d_row_sample,
                            void* stream) {
  nt_status st = check_partition(part, false);
  if (st != NT_OK) return st;
  if (!d_row_start || (part->T > 0 && !d_row_sample))
    return fail(NT_ERR_INVALID, "NULL row split pointer");
  if (!aligned16(d_row_start) || !aligned16(d_row_sample))
    return fail(NT_ERR_INVALID, "pointers must be 16-byte aligned");
  cudaError_t e = launch_partition_rows(part->lengths, part->col_lengths, part->cu_seqlens, part->pair_off,
                                        part->B, part->T, part->P, d_row_start, d_row_sample,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "partition rows launch");
  part->row_start = d_row_start;
  part->row_sample = d_row_sample;
  return NT_OK;
}

size_t nt_pair_broadcast_workspace_bytes(int64_t T, int32_t C_z) {
  if (T < 0 || C_z < 0) return 0;
  return (size_t)2 * (size_t)T * (size_t)C_z * sizeof(float);
}

size_t nt_pair_broadcast_workspace_bytes_rect(int64_t T_rows, int64_t T_cols, int32_t C_z) {
  if (T_rows < 0 || T_cols < 0 || C_z < 0) return 0;
  return (size_t)(T_rows + T_cols) * (size_t)C_z * sizeof(float);
}

nt_status nt_pair_broadcast(const nt_partition* part, nt_dtype dtype, const void* s_left,
                            const void* s_right, int32_t C_s, const void* W_a, const void* W_b,
                            int32_t C_z, void* z, void* workspace, size_t workspace_bytes,
                            void* stream) {
  nt_status st = check_partition(part, true);
  if (st != NT_OK) return st;
  if (!dtype_ok(dtype)) return fail(NT_ERR_INVALID, "bad dtype %d", (int)dtype);
  if (!width_ok(dtype, C_s) || !width_ok(dtype, C_z))
    return fail(NT_ERR_UNSUPPORTED, "C_s=%d, C_z=%d must be positive multiples of %d", C_s, C_z,
                dtype == NT_BF16 ? 8 : 4);
  const int64_t T_cols = t_cols_of(part);
  const size_t need = nt_pair_broadcast_workspace_bytes_rect(part->T, T_cols, C_z);
  // an array of no elements may be NULL (an empty batch)
  if (!W_a || !W_b || (part->T > 0 && !s_left) || (T_cols > 0 && !s_right) || (part->P > 0 && !z) ||
      (need > 0 && !workspace))
    return fail(NT_ERR_INVALID, "NULL pointer");
  if (!aligned16(s_left) || !aligned16(s_right) || !aligned16(W_a) || !aligned16(W_b) ||
      !aligned16(z) || !aligned16(workspace))
    return fail(NT_ERR_INVALID, "pointers must be 16-byte aligned");
  if (workspace_bytes < need)
    return fail(NT_ERR_INVALID, "workspace of %zu bytes < %zu needed", workspace_bytes, need);
  if (part->T == 0) return NT_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* u = static_cast<float*>(workspace);
  float* v = u + part->T * (int64_t)C_z;
  cudaError_t e = project_uv(part, dtype, s_left, s_right, C_s, W_a, W_b, C_z, u, v, s);
  if (e != cudaSuccess) return cuda_fail(e, "projection launch");
  e = launch_broadcast(dtype, u, v, part, C_z, z, s);
  if (e != cudaSuccess) return cuda_fail(e, "broadcast launch");
  return NT_OK;
}

nt_status nt_pair_transition(const nt_partition* part, nt_dtype dtype, const void* z_in,
                             void* z_out, int32_t C_z, int32_t H_t, const float* ln_gamma,
                             const float* ln_beta, float ln_eps, const void* W1,
                             const float* b1, const void* W2, const float* b2, void* stream) {
  return pair_transition(part, dtype, z_in, z_out, C_z, H_t, ln_gamma, ln_beta, ln_eps, W1, b1, nullptr, nullptr,
                         W2, b2, stream);
}

nt_status nt_pair_transition_swiglu(const nt_partition* part, nt_dtype dtype, const void* z_in, void* z_out,
                                    int32_t C_z, int32_t H_t, const float* ln_gamma, const float* ln_beta,
                                    float ln_eps, const void* W1, const float* b1, const void* W3,
                                    const float* b3, const void* W2, const float* b2, void* stream) {
  if (!W3) return fail(NT_ERR_INVALID, "W3 (the value projection) is NULL");
  return pair_transition(part, dtype, z_in, z_out, C_z, H_t, ln_gamma, ln_beta, ln_eps, W1, b1, W3, b3, W2, b2,
                         stream);
}

nt_status nt_pair_transition_cells(int64_t n_cells, nt_dtype dtype, const void* z_in, void* z_out, int32_t C_z,
                                   int32_t H_t, const float* ln_gamma, const float* ln_beta, float ln_eps,
                                   const void* W1, const float* b1, const void* W3, const float* b3,
                                   const void* W2, const float* b2, void* stream) {
  return transition_cells(n_cells, dtype, z_in, z_out, C_z, H_t, ln_gamma, ln_beta, ln_eps, W1, b1, W3, b3, W2,
                          b2, stream);
}

nt_status nt_pair_reduce(const nt_partition* part, nt_dtype dtype, const void* z, int32_t C_z,
                         void* m, const void* W_g, const float* b_g, const void* s_in,
                         void* s_out, int32_t C_s, void* stream) {
  nt_status st = check_partition(part, true);
  if (st != NT_OK) return st;
  if (!dtype_ok(dtype)) return fail(NT_ERR_INVALID, "bad dtype %d", (int)dtype);
  if (!width_ok(dtype, C_z)) return fail(NT_ERR_UNSUPPORTED, "C_z=%d", C_z);
  if (dtype == NT_BF16 && C_z > 1024) return fail(NT_ERR_UNSUPPORTED, "bf16 C_z=%d > 1024", C_z);
  if ((part->P > 0 && !z) || (part->T > 0 && !m)) return fail(NT_ERR_INVALID, "NULL pointer");
  if (W_g && ((part->T > 0 && !s_out) || !width_ok(dtype, C_s)))
    return fail(NT_ERR_INVALID, "W_g given: s_out must be set and C_s=%d valid", C_s);
  if (!aligned16(z) || !aligned16(m) || !aligned16(W_g) || !aligned16(b_g) || !aligned16(s_in) ||
      !aligned16(s_out))
    return fail(NT_ERR_INVALID, "pointers must be 16-byte aligned");
  if (part->T == 0) return NT_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_reduce(dtype, z, part, C_z, m, s);
  if (e != cudaSuccess) return cuda_fail(e, "reduce launch");
  if (W_g) {
    LinearProblem prob = {m, W_g, b_g, s_in, s_out};
    e = linear_tc_supported(dtype, part->T, C_s, C_z)
            ? launch_linear_tc(0, &prob, 1, part->T, C_s, C_z, status_word(), s)
            : launch_linear(dtype, dtype == NT_F32, &prob, 1, part->T, C_s, C_z, s);
    if (e != cudaSuccess) return cuda_fail(e, "g projection launch");
  }
  return NT_OK;
}

size_t nt_pair_reduce_loss_workspace_bytes(void) {
  return ((eq5_loss_workspace_bytes() + 255) & ~(size_t)255) + (size_t)kReduceMaxGrid * sizeof(double);
}

nt_status nt_pair_reduce_loss(const nt_partition* part, nt_dtype dtype, const void* z, int32_t C_z, void* m,
                              const void* W_g, const float* b_g, const void* s_in, void* s_out, int32_t C_s,
                              float* d_loss, void* workspace, size_t workspace_bytes, void* stream) {
  nt_status st = check_partition(part, true);
  if (st != NT_OK) return st;
  if (!dtype_ok(dtype)) return fail(NT_ERR_INVALID, "bad dtype %d", (int)dtype);
  if (!width_ok(dtype, C_z) || !width_ok(dtype, C_s)) return fail(NT_ERR_UNSUPPORTED, "C_z=%d, C_s=%d", C_z, C_s);
  if (dtype == NT_BF16 && C_z > 1024) return fail(NT_ERR_UNSUPPORTED, "bf16 C_z=%d > 1024", C_z);
  if (!W_g || !d_loss || !workspace || (part->P > 0 && !z) || (part->T > 0 && (!m || !s_out)))
    return fail(NT_ERR_INVALID, "NULL pointer");
  if (!aligned16(z) || !aligned16(m) || !aligned16(W_g) || !aligned16(b_g) || !aligned16(s_in) ||
      !aligned16(s_out) || !aligned16(workspace))
    return fail(NT_ERR_INVALID, "pointers must be 16-byte aligned");
  const size_t need = nt_pair_reduce_loss_workspace_bytes();
  if (workspace_bytes < need) return fail(NT_ERR_INVALID, "workspace of %zu bytes < %zu needed", workspace_bytes, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  double* partial = static_cast<double*>(workspace);
  double* pair_sq = reinterpret_cast<double*>(static_cast<uint8_t*>(workspace) +
                                              ((eq5_loss_workspace_bytes() + 255) & ~(size_t)255));
  const bool fused = reduce_sq_supported(C_z);
  int npair = 0;
  cudaError_t e = launch_reduce(dtype, z, part, C_z, m, s, fused ? pair_sq : nullptr, &npair);
  if (e != cudaSuccess) return cuda_fail(e, "reduce launch");
  if (part->T > 0) {
    LinearProblem prob = {m, W_g, b_g, s_in, s_out};
    e = linear_tc_supported(dtype, part->T, C_s, C_z)
            ? launch_linear_tc(0, &prob, 1, part->T, C_s, C_z, status_word(), s)
            : launch_linear(dtype, dtype == NT_F32, &prob, 1, part->T, C_s, C_z, s);
    if (e != cudaSuccess) return cuda_fail(e, "g projection launch");
  }
  e = fused ? launch_eq5_loss_rows(dtype, part, s_out, C_s, C_z, d_loss, pair_sq, npair, partial, s)
            : launch_eq5_loss(dtype, part, s_out, C_s, z, C_z, d_loss, nullptr, nullptr, partial, s);
  if (e != cudaSuccess) return cuda_fail(e, "loss launch");
  return NT_OK;
}

size_t nt_pair_block_fused_workspace_bytes(int64_t T, int64_t T_cols, int32_t C_z) {
  if (T < 0 || T_cols < 0 || C_z < 0) return 0;
  return (size_t)(2 * T + T_cols) * (size_t)C_z * sizeof(float);
}

nt_status nt_pair_block_fused(const nt_partition* part, nt_dtype dtype, const void* s_left, const void* s_right,
                              int32_t C_s, const void* W_a, const void* W_b, int32_t C_z, int32_t H_t,
                              const float* ln_gamma, const float* ln_beta, float ln_eps, const void* W1,
                              const float* b1, const void* W3, const float* b3, const void* W2, const float* b2,
                              const void* W_g, const float* b_g, void* z_out, void* m, void* s_out,
                              void* workspace, size_t workspace_bytes, void* stream) {
  nt_status st = check_partition(part, true);
  if (st != NT_OK) return st;
  if (!dtype_ok(dtype)) return fail(NT_ERR_INVALID, "bad dtype %d", (int)dtype);
  if (!width_ok(dtype, C_s) || !width_ok(dtype, C_z) || !width_ok(dtype, H_t))
    return fail(NT_ERR_UNSUPPORTED, "C_s=%d, C_z=%d, H_t=%d must be positive multiples of %d", C_s, C_z, H_t,
                dtype == NT_BF16 ? 8 : 4);
  // an array of no elements may be NULL (an empty batch)
  const int64_t T_cols_f = t_cols_of(part);
  if (!W_a || !W_b || !ln_gamma || !ln_beta || !W1 || !W2 || (part->T > 0 && (!s_left || !m)) ||
      (T_cols_f > 0 && !s_right) || (part->P > 0 && !z_out) ||
      (nt_pair_block_fused_workspace_bytes(part->T, T_cols_f, C_z) > 0 && !workspace))
    return fail(NT_ERR_INVALID, "NULL pointer");
  if (W_g && part->T > 0 && !s_out) return fail(NT_ERR_INVALID, "W_g given: s_out must be set");
  if (!aligned16(s_left) || !aligned16(s_right) || !aligned16(W_a) || !aligned16(W_b) || !aligned16(W1) ||
      !aligned16(W2) || !aligned16(W3) || !aligned16(z_out) || !aligned16(m) || !aligned16(workspace) ||
      !aligned16(W_g) || !aligned16(s_out) || !aligned16(ln_gamma) || !aligned16(ln_beta) || !aligned16(b1) ||
      !aligned16(b2) || !aligned16(b3) || !aligned16(b_g))
    return fail(NT_ERR_INVALID, "pointers must be 16-byte aligned");
  if (!(ln_eps >= 0.0f)) return fail(NT_ERR_INVALID, "ln_eps must be >= 0");
  if (part->P > kMaxCells)
    return fail(NT_ERR_OVERFLOW, "%lld cells: at most %lld", (long long)part->P, (long long)kMaxCells);
  const int64_t T_cols = t_cols_of(part);
  const size_t need = nt_pair_block_fused_workspace_bytes(part->T, T_cols, C_z);
  if (workspace_bytes < need)
    return fail(NT_ERR_INVALID, "workspace of %zu bytes < %zu needed", workspace_bytes, need);
  if (part->T == 0) return NT_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!transition_tc_supported(dtype, C_z, H_t, W3 != nullptr)) {
    // the same block through the three pair calls' kernels
    st = nt_pair_broadcast(part, dtype, s_left, s_right, C_s, W_a, W_b, C_z, z_out, workspace, workspace_bytes,
                           stream);
    if (st != NT_OK) return st;
    st = W3 ? nt_pair_transition_swiglu(part, dtype, z_out, z_out, C_z, H_t, ln_gamma, ln_beta, ln_eps, W1, b1, W3,
                                        b3, W2, b2, stream)
            : nt_pair_transition(part, dtype, z_out, z_out, C_z, H_t, ln_gamma, ln_beta, ln_eps, W1, b1, W2, b2,
                                 stream);
    if (st != NT_OK) return st;
    return nt_pair_reduce(part, dtype, z_out, C_z, m, W_g, b_g, s_left, s_out, C_s, stream);
  }
  float* u = static_cast<float*>(workspace);
  float* v = u + part->T * (int64_t)C_z;
  float* m_acc = v + T_cols * (int64_t)C_z;
  cudaError_t e = project_uv(part, dtype, s_left, s_right, C_s, W_a, W_b, C_z, u, v, s);
  if (e != cudaSuccess) return cuda_fail(e, "projection launch");
  e = cudaMemsetAsync(m_acc, 0, (size_t)part->T * C_z * sizeof(float), s);
  if (e != cudaSuccess) return cuda_fail(e, "row-sum clear");
  if (part->P > 0) {
    e = launch_block_fused_tc(u, v, part, z_out, C_z, H_t, ln_gamma, ln_beta, ln_eps, W1, b1, W3, b3, W2, b2, m_acc,
                              status_word(), s);
    if (e != cudaSuccess) return cuda_fail(e, "fused block launch");
  }
  e = launch_mean_finish(dtype, m_acc, part, C_z, m, s);
  if (e != cudaSuccess) return cuda_fail(e, "row mean launch");
  if (W_g) {
    LinearProblem prob = {m, W_g, b_g, s_left, s_out};
    e = linear_tc_supported(dtype, part->T, C_s, C_z)
            ? launch_linear_tc(0, &prob, 1, part->T, C_s, C_z, status_word(), s)
            : launch_linear(dtype, dtype == NT_F32, &prob, 1, part->T, C_s, C_z, s);
    if (e != cudaSuccess) return cuda_fail(e, "g projection launch");
  }
  return NT_OK;
}

size_t nt_varlen_attn_workspace_bytes(void) { return kAttnWorkBytes; }

nt_status nt_varlen_attn_qk(nt_dtype dtype, const void* q, const void* k, const void* v,
                            const int32_t* d_cu_seqlens_q, const int32_t* d_cu_seqlens_k, int32_t B,
                            int64_t T_q, int64_t T_k, int32_t max_len_q, int32_t H, int32_t d, float scale,
                            int32_t causal, void* o, float* lse, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (!dtype_ok(dtype)) return fail(NT_ERR_INVALID, "bad dtype %d", (int)dtype);
  if (B < 0 || T_q < 0 || T_k < 0 || H <= 0 || d <= 0 || max_len_q < 0)
    return fail(NT_ERR_INVALID, "bad sizes B=%d T_q=%lld T_k=%lld H=%d d=%d max_len_q=%d", B, (long long)T_q,
                (long long)T_k, H, d, max_len_q);
  if (!(scale > 0.f) || std::isinf(scale)) return fail(NT_ERR_INVALID, "scale must be finite and > 0");
  if (causal != 0 && causal != 1) return fail(NT_ERR_INVALID, "causal must be 0 or 1");
  if (T_q > 0x7fffffffLL || T_k > 0x7fffffffLL)
    return fail(NT_ERR_OVERFLOW, "T_q = %lld, T_k = %lld: token counts must fit int32", (long long)T_q,
                (long long)T_k);
  if (T_q > 0 && B == 0) return fail(NT_ERR_INVALID, "T_q > 0 with no segments");
  if (T_q > 0 && (!q || !o || !d_cu_seqlens_q || !d_cu_seqlens_k)) return fail(NT_ERR_INVALID, "NULL pointer");
  if (T_q > 0 && T_k > 0 && (!k || !v)) return fail(NT_ERR_INVALID, "NULL key or value pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(workspace))
    return fail(NT_ERR_INVALID, "pointers must be 16-byte aligned");
  if (workspace && workspace_bytes < kAttnWorkBytes)
    return fail(NT_ERR_INVALID, "workspace of %zu bytes < %zu needed", workspace_bytes, kAttnWorkBytes);
  if (T_q == 0) return NT_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const AttnProblem prob = {q, k, v, d_cu_seqlens_q, d_cu_seqlens_k, B, T_q, T_k, max_len_q,
                            H, d, scale, causal != 0, o, lse, static_cast<unsigned int*>(workspace)};
  cudaError_t e;
  if (attn_tc_supported(dtype, d) && T_k > 0) {
    e = launch_attn_tc(prob, status_word(), s);
    if (e != cudaSuccess) return cuda_fail(e, "varlen attention (tensor core) launch");
    return NT_OK;
  }
  if (!attn_simt_supported(d)) return fail(NT_ERR_UNSUPPORTED, "head width d=%d", d);
  e = launch_attn_simt(dtype, prob, status_word(), s);
  if (e != cudaSuccess) return cuda_fail(e, "varlen attention launch");
  return NT_OK;
}

size_t nt_varlen_attn_bwd_workspace_bytes(int64_t T_q, int32_t H) {
  if (T_q < 0 || H < 0) return 0;
  return bwd_counter_offset(T_q, H) + kAttnWorkBytes;
}

nt_status nt_varlen_attn_bwd(nt_dtype dtype, const void* q, const void* k, const void* v, const void* o,
                             const void* d_o, const float* lse, const int32_t* d_cu_seqlens_q,
                             const int32_t* d_cu_seqlens_k, int32_t B, int64_t T_q, int64_t T_k,
                             int32_t max_len_q, int32_t max_len_k, int32_t H, int32_t d, float scale,
                             int32_t causal, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (!dtype_ok(dtype)) return fail(NT_ERR_INVALID, "bad dtype %d", (int)dtype);
  if (B < 0 || T_q < 0 || T_k < 0 || H <= 0 || d <= 0 || max_len_q < 0 || max_len_k < 0)
    return fail(NT_ERR_INVALID, "bad sizes B=%d T_q=%lld T_k=%lld H=%d d=%d max_len_q=%d max_len_k=%d", B,
                (long long)T_q, (long long)T_k, H, d, max_len_q, max_len_k);
  if (!(scale > 0.f) || std::isinf(scale)) return fail(NT_ERR_INVALID, "scale must be finite and > 0");
  if (causal != 0 && causal != 1) return fail(NT_ERR_INVALID, "causal must be 0 or 1");
  if (T_q > 0x7fffffffLL || T_k > 0x7fffffffLL)
    return fail(NT_ERR_OVERFLOW, "T_q = %lld, T_k = %lld: token counts must fit int32", (long long)T_q,
                (long long)T_k);
  if ((T_q > 0 || T_k > 0) && B == 0) return fail(NT_ERR_INVALID, "tokens with no segments");
  if (!attn_bwd_supported(d)) return fail(NT_ERR_UNSUPPORTED, "head width d=%d", d);
  if (T_q > 0 && (!q || !o || !d_o || !lse || !dq || !workspace || !d_cu_seqlens_q || !d_cu_seqlens_k))
    return fail(NT_ERR_INVALID, "NULL pointer");
  if (T_k > 0 && (!k || !v || !dk || !dv || !d_cu_seqlens_q || !d_cu_seqlens_k))
    return fail(NT_ERR_INVALID, "NULL key-side pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(d_o) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
    return fail(NT_ERR_INVALID, "pointers must be 16-byte aligned");
  if (workspace_bytes < nt_varlen_attn_bwd_workspace_bytes(T_q, H))
    return fail(NT_ERR_INVALID, "workspace of %zu bytes < %zu needed", workspace_bytes,
                nt_varlen_attn_bwd_workspace_bytes(T_q, H));
  if (T_q == 0 && T_k == 0) return NT_OK;
  const AttnBwdProblem prob = {q, k, v, o, d_o, lse, d_cu_seqlens_q, d_cu_seqlens_k, B, T_q, T_k,
                               max_len_q, max_len_k, H, d, scale, causal != 0, dq, dk, dv,
                               reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(workspace) +
                                                               bwd_counter_offset(T_q, H))};
  cudaError_t e = launch_attn_bwd(dtype, prob, static_cast<float*>(workspace), status_word(),
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "varlen attention backward launch");
  return NT_OK;
}

nt_status nt_varlen_attn(nt_dtype dtype, const void* q, const void* k, const void* v,
                         const int32_t* d_cu_seqlens, int32_t B, int64_t T, int32_t max_len,
                         int32_t H, int32_t d, float scale, void* o, float* lse, void* workspace,
                         size_t workspace_bytes, void* stream) {
  return nt_varlen_attn_qk(dtype, q, k, v, d_cu_seqlens, d_cu_seqlens, B, T, T, max_len, H, d, scale, 0, o,
                           lse, workspace, workspace_bytes, stream);
}

size_t nt_pair_block_loss_workspace_bytes(void) { return eq5_loss_workspace_bytes(); }

nt_status nt_pair_block_loss(const nt_partition* part, nt_dtype dtype, const void* s_out, int32_t C_s,
                             const void* z_tilde, int32_t C_z, float* d_loss, float* ds_out, float* dz_tilde,
                             void* workspace, size_t workspace_bytes, void* stream) {
  nt_status st = check_partition(part, true);
  if (st != NT_OK) return st;
  if (!dtype_ok(dtype)) return fail(NT_ERR_INVALID, "bad dtype %d", (int)dtype);
  if (!width_ok(dtype, C_s) || !width_ok(dtype, C_z))
    return fail(NT_ERR_UNSUPPORTED, "C_s=%d, C_z=%d must be positive multiples of %d", C_s, C_z,
                dtype == NT_BF16 ? 8 : 4);
  if (!d_loss || !workspace || (part->T > 0 && !s_out) || (part->P > 0 && !z_tilde))
    return fail(NT_ERR_INVALID, "NULL pointer");
  if (!aligned16(s_out) || !aligned16(z_tilde) || !aligned16(ds_out) || !aligned16(dz_tilde) ||
      !aligned16(workspace))
    return fail(NT_ERR_INVALID, "pointers must be 16-byte aligned");
  if (workspace_bytes < eq5_loss_workspace_bytes())
    return fail(NT_ERR_INVALID, "workspace of %zu bytes < %zu needed", workspace_bytes, eq5_loss_workspace_bytes());
  cudaError_t e = launch_eq5_loss(dtype, part, s_out, C_s, z_tilde, C_z, d_loss, ds_out, dz_tilde, workspace,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "loss launch");
  return NT_OK;
}

size_t nt_pair_block_backward_workspace_bytes(nt_dtype dtype, int64_t T, int64_t P, int32_t C_z, int32_t H_t) {
  if (T < 0 || P < 0 || C_z < 0 || H_t < 0) return 0;
  return block_bwd_workspace_bytes(dtype, T, P, C_z, H_t);
}

nt_status nt_pair_block_backward(const nt_partition* part, nt_dtype dtype, const void* s, int32_t C_s,
                                 const void* W_a, const void* W_b, int32_t C_z, int32_t H_t, const float* ln_gamma,
                                 const float* ln_beta, float ln_eps, const void* W1, const float* b1, const void* W2,
                                 const void* W_g, const void* m, const float* ds_out, const float* dz_tilde,
                                 float* ds, float* dW_a, float* dW_b, float* dgamma, float* dbeta, float* dW1,
                                 float* db1, float* dW2, float* db2, float* dW_g, float* db_g, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  nt_status st = check_block_backward(part, dtype, C_s, C_z, H_t, ln_eps);
  if (st != NT_OK) return st;
  if (!W_a || !W_b || !ln_gamma || !ln_beta || !W1 || !W2 || !W_g || !dW_a || !dW_b || !dgamma || !dbeta ||
      !dW1 || !db1 || !dW2 || !db2 || !dW_g || !db_g || !workspace)
    return fail(NT_ERR_INVALID, "NULL pointer");
  if (part->T > 0 && (!s || !m || !ds_out || !ds)) return fail(NT_ERR_INVALID, "NULL single-row pointer");
  const void* ptrs[] = {s, W_a, W_b, ln_gamma, ln_beta, W1, b1, W2, W_g, m, ds_out, dz_tilde, ds, dW_a, dW_b,
                        dgamma, dbeta, dW1, db1, dW2, db2, dW_g, db_g, workspace};
  for (const void* q : ptrs)
    if (!aligned16(q)) return fail(NT_ERR_INVALID, "pointers must be 16-byte aligned");
  const size_t need = nt_pair_block_backward_workspace_bytes(dtype, part->T, part->P, C_z, H_t);
  if (workspace_bytes < need) return fail(NT_ERR_INVALID, "workspace of %zu bytes < %zu needed", workspace_bytes, need);
  return block_backward_run(part, dtype, s, C_s, W_a, W_b, C_z, H_t, ln_gamma, ln_beta, ln_eps, W1, b1, W2, W_g, m,
                            ds_out, dz_tilde, nullptr, ds, dW_a, dW_b, dgamma, dbeta, dW1, db1, dW2, db2, dW_g, db_g,
                            workspace, static_cast<cudaStream_t>(stream));
}

size_t nt_pair_block_loss_backward_workspace_bytes(nt_dtype dtype, int64_t T, int64_t P, int32_t C_s, int32_t C_z,
                                                   int32_t H_t) {
  if (T < 0 || P < 0 || C_s < 0 || C_z < 0 || H_t < 0) return 0;
  return loss_bwd_layout(dtype, T, P, C_s, C_z, H_t).end;
}

nt_status nt_pair_block_loss_backward(const nt_partition* part, nt_dtype dtype, const void* s, int32_t C_s,
                                      const void* W_a, const void* W_b, int32_t C_z, int32_t H_t,
                                      const float* ln_gamma, const float* ln_beta, float ln_eps, const void* W1,
                                      const float* b1, const void* W2, const void* W_g, const void* m,
                                      const void* s_out, const void* z_tilde, float* d_loss, float* ds, float* dW_a,
                                      float* dW_b, float* dgamma, float* dbeta, float* dW1, float* db1, float* dW2,
                                      float* db2, float* dW_g, float* db_g, void* workspace, size_t workspace_bytes,
                                      void* stream) {
  nt_status st = check_block_backward(part, dtype, C_s, C_z, H_t, ln_eps);
  if (st != NT_OK) return st;
  if (!W_a || !W_b || !ln_gamma || !ln_beta || !W1 || !W2 || !W_g || !dW_a || !dW_b || !dgamma || !dbeta ||
      !dW1 || !db1 || !dW2 || !db2 || !dW_g || !db_g || !d_loss || !workspace)
    return fail(NT_ERR_INVALID, "NULL pointer");
  if (part->T > 0 && (!s || !m || !s_out || !ds)) return fail(NT_ERR_INVALID, "NULL single-row pointer");
  if (part->P > 0 && !z_tilde) return fail(NT_ERR_INVALID, "NULL z_tilde");
  const void* ptrs[] = {s, W_a, W_b, ln_gamma, ln_beta, W1, b1, W2, W_g, m, s_out, z_tilde, ds, dW_a, dW_b,
                        dgamma, dbeta, dW1, db1, dW2, db2, dW_g, db_g, workspace};
  for (const void* q : ptrs)
    if (!aligned16(q)) return fail(NT_ERR_INVALID, "pointers must be 16-byte aligned");
  const LossBwdLayout L = loss_bwd_layout(dtype, part->T, part->P, C_s, C_z, H_t);
  if (workspace_bytes < L.end) return fail(NT_ERR_INVALID, "workspace of %zu bytes < %zu needed", workspace_bytes, L.end);
  cudaStream_t st_ = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  float* dx = reinterpret_cast<float*>(w + L.dx);
  const bool tc = block_bwd_tc(dtype, part->P, C_z, H_t);
  // the loss and dX~; dL/dz~ only where the backward does not form it from z~
  float* dz = tc ? nullptr : reinterpret_cast<float*>(w + L.dz);
  cudaError_t e = launch_eq5_loss(dtype, part, s_out, C_s, z_tilde, C_z, d_loss, part->T > 0 ? dx : nullptr,
                                  part->P > 0 ? dz : nullptr, w, st_);
  if (e != cudaSuccess) return cuda_fail(e, "loss launch");
  return block_backward_run(part, dtype, s, C_s, W_a, W_b, C_z, H_t, ln_gamma, ln_beta, ln_eps, W1, b1, W2, W_g, m,
                            dx, tc ? nullptr : dz, tc ? z_tilde : nullptr, ds, dW_a, dW_b, dgamma, dbeta, dW1, db1,
                            dW2, db2, dW_g, db_g, w + L.bwd, st_);
}

nt_status nt_selftest_bounded_wait(int32_t mode, uint64_t delay_ns, uint64_t limit_ns, int64_t* d_result,
                                   void* stream) {
  if (mode < 0 || mode > 2) return fail(NT_ERR_INVALID, "mode %d (0, 1 or 2)", mode);
  if (limit_ns == 0 || limit_ns > kSelftestMaxNs || delay_ns > kSelftestMaxNs)
    return fail(NT_ERR_INVALID, "limit_ns must be in (0, 2 s] and delay_ns at most 2 s");
  if (!d_result) return fail(NT_ERR_INVALID, "NULL pointer");
  if ((reinterpret_cast<uintptr_t>(d_result) & 7u) != 0) return fail(NT_ERR_INVALID, "d_result must be 8-byte aligned");
  unsigned int* status = status_word();
  if (!status) return fail(NT_ERR_CUDA, "device status word not available");
  const cudaError_t e = launch_selftest_wait(mode, delay_ns, limit_ns, d_result, status,
                                             static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return NT_OK;
}

nt_status nt_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  unsigned int word = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&word, g_device_status, sizeof(word));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_fail(e, "device status readback");
  if (word & kDevTimeout) return fail(NT_ERR_TIMEOUT, "a bounded device wait ran out (word 0x%x)", word);
  if (word & kDevCheck) return fail(NT_ERR_DEVICE_CHECK, "a device-side data check failed (word 0x%x)", word);
  return NT_OK;
}

}  // extern "C"
