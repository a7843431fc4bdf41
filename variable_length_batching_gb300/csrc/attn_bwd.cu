// Backward of variable-length attention ("Variable-length attention and data
// packing", "What it is" / "How it works", with the causal and cross forms of
// nt_varlen_attn_qk) on CUDA cores: for the upstream gradient dO and the
// forward's natural-log LSE, per segment and head,
//     P  = exp(scale Q K^T - lse)                (recomputed, masked as forward)
//     dV = P^T dO,  dS = P * (dO V^T - D),  D = rowsum(dO * O)
//     dQ = scale dS K,  dK = scale dS^T Q
// Three kernels, each a warp per token row and head (lane l holds features
// l, l + 32, ...; dot products are warp butterflies): D per query row, then
// dQ walking the row's visible keys, then dK and dV walking the queries that
// see each key.  No atomics: every output row has exactly one owner.  For
// bf16 with d = 64, the tensor-core kernels run instead (attn_bwd_tc.cu),
// their dQ kernel forming D itself.
#include <type_traits>

#include "nt_common.cuh"

namespace nt {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// last segment b with cu[b] <= t (t inside [cu[0], cu[B]))
__device__ __forceinline__ int segment_of(const int32_t* __restrict__ cu, int B, int64_t t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One warp per token: the token's rows of O and dO for all H heads are
// H * D contiguous elements, read as 16-byte chunks with consecutive lanes
// on consecutive chunks (lane l takes chunks l, l + 32, ...).  A head's
// D / kVec chunks sit in consecutive lanes of one pass (kVec divides D and
// D / kVec divides 32), so a butterfly over those lanes finishes the head's
// sum and its first lane writes D[h, t] in the [H, T_q] layout.
template <typename T, int D>
__global__ void __launch_bounds__(256)
rowdot_kernel(const T* __restrict__ o, const T* __restrict__ d_o, int64_t Tq, int H, float* __restrict__ Dbuf) {
  constexpr int kVec = 16 / (int)sizeof(T);          // elements per 16-byte chunk
  constexpr int kCph = D / kVec;                      // chunks per head: 2 .. 32
  static_assert(32 % kCph == 0, "a head's chunks must not straddle two passes");
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= Tq) return;                                // warp-uniform
  const uint4* po = reinterpret_cast<const uint4*>(o + t * H * D);
  const uint4* pd = reinterpret_cast<const uint4*>(d_o + t * H * D);
  const int chunks = H * kCph;
  for (int base = 0; base < chunks; base += 32) {     // warp-uniform trip count
    const int c = base + lane;
    float acc[2] = {0.f, 0.f};
    if (c < chunks) {
      const uint4 a = po[c], b = pd[c];
      const T* ea = reinterpret_cast<const T*>(&a);
      const T* eb = reinterpret_cast<const T*>(&b);
#pragma unroll
      for (int e = 0; e < kVec; ++e) acc[e & 1] = fmaf(to_f32(eb[e]), to_f32(ea[e]), acc[e & 1]);
    }
    float sum = acc[0] + acc[1];
#pragma unroll
    for (int off = 1; off < kCph; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (c < chunks && (lane % kCph) == 0) Dbuf[(int64_t)(c / kCph) * Tq + t] = sum;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
dq_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, const T* __restrict__ d_o,
          const float* __restrict__ lse, const float* __restrict__ Dbuf, const int32_t* __restrict__ cu_q,
          const int32_t* __restrict__ cu_k, int B, int64_t Tq, int64_t Tk, int H, float scale, bool causal,
          T* __restrict__ dq, unsigned int* status) {
  constexpr int kPer = D / 32;
  const int64_t w = (int64_t)blockIdx.x * kWarps + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (w >= Tq * H) return;
  const int64_t t = w / H;
  const int h = (int)(w % H);
  const int b = segment_of(cu_q, B, t);
  const int qlo = cu_q[b], qhi = cu_q[b + 1], klo = cu_k[b], khi = cu_k[b + 1];
  float acc[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) acc[u] = 0.f;
  if (qlo < 0 || qlo > t || qhi <= t || qhi > Tq || klo < 0 || khi < klo || khi > Tk) {
    if (lane == 0) flag_device(status, kDevCheck);
    return;
  }
  const float l = lse[(int64_t)h * Tq + t];
  int64_t kend = khi;
  if (causal) kend = max((int64_t)klo, min((int64_t)khi, (int64_t)klo + (t - qlo) + (khi - klo) - (qhi - qlo) + 1));
  if (l != -INFINITY) {
    float qv[kPer], dov[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int64_t idx = (t * H + h) * D + lane + 32 * u;
      qv[u] = to_f32(q[idx]);
      dov[u] = to_f32(d_o[idx]);
    }
    const float Dt = Dbuf[(int64_t)h * Tq + t];
    for (int64_t j = klo; j < kend; ++j) {
      float kv[kPer], vv[kPer], s = 0.f, dp = 0.f;
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int64_t idx = (j * H + h) * D + lane + 32 * u;
        kv[u] = to_f32(k[idx]);
        vv[u] = to_f32(v[idx]);
        s = fmaf(qv[u], kv[u], s);
        dp = fmaf(dov[u], vv[u], dp);
      }
      s = warp_sum(s);
      dp = warp_sum(dp);
      const float p = expf(s * scale - l);
      const float ds = p * (dp - Dt);
#pragma unroll
      for (int u = 0; u < kPer; ++u) acc[u] = fmaf(ds, kv[u], acc[u]);
    }
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) dq[(t * H + h) * D + lane + 32 * u] = from_f32<T>(acc[u] * scale);
}

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
dkv_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, const T* __restrict__ d_o,
           const float* __restrict__ lse, const float* __restrict__ Dbuf, const int32_t* __restrict__ cu_q,
           const int32_t* __restrict__ cu_k, int B, int64_t Tq, int64_t Tk, int H, float scale, bool causal,
           T* __restrict__ dk, T* __restrict__ dv, unsigned int* status) {
  constexpr int kPer = D / 32;
  const int64_t w = (int64_t)blockIdx.x * kWarps + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (w >= Tk * H) return;
  const int64_t j = w / H;
  const int h = (int)(w % H);
  const int b = segment_of(cu_k, B, j);
  const int qlo = cu_q[b], qhi = cu_q[b + 1], klo = cu_k[b], khi = cu_k[b + 1];
  float gk[kPer], gv[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) { gk[u] = 0.f; gv[u] = 0.f; }
  if (klo < 0 || klo > j || khi <= j || khi > Tk || qlo < 0 || qhi < qlo || qhi > Tq) {
    if (lane == 0) flag_device(status, kDevCheck);
    return;
  }
  // causal: query i (of the segment) sees local key jj when jj <= i + (n_k - n_q)
  int64_t istart = qlo;
  if (causal) istart = max((int64_t)qlo, (int64_t)qlo + (j - klo) - ((khi - klo) - (qhi - qlo)));
  float kv[kPer], vv[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int64_t idx = (j * H + h) * D + lane + 32 * u;
    kv[u] = to_f32(k[idx]);
    vv[u] = to_f32(v[idx]);
  }
  for (int64_t i = istart; i < qhi; ++i) {
    const float l = lse[(int64_t)h * Tq + i];
    if (l == -INFINITY) continue;           // a query that sees no key: no gradient
    float qv[kPer], dov[kPer], s = 0.f, dp = 0.f;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int64_t idx = (i * H + h) * D + lane + 32 * u;
      qv[u] = to_f32(q[idx]);
      dov[u] = to_f32(d_o[idx]);
      s = fmaf(qv[u], kv[u], s);
      dp = fmaf(dov[u], vv[u], dp);
    }
    s = warp_sum(s);
    dp = warp_sum(dp);
    const float p = expf(s * scale - l);
    const float ds = p * (dp - Dbuf[(int64_t)h * Tq + i]);
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      gv[u] = fmaf(p, dov[u], gv[u]);
      gk[u] = fmaf(ds, qv[u], gk[u]);
    }
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int64_t idx = (j * H + h) * D + lane + 32 * u;
    dk[idx] = from_f32<T>(gk[u] * scale);
    dv[idx] = from_f32<T>(gv[u]);
  }
}

template <typename T, int D>
cudaError_t launch_d(const AttnBwdProblem& p, float* Dbuf, unsigned int* status, cudaStream_t s) {
  const int64_t wq = p.T_q * p.H, wk = p.T_k * p.H;
  const unsigned gq = (unsigned)((wq + kWarps - 1) / kWarps), gk = (unsigned)((wk + kWarps - 1) / kWarps);
  // the tensor-core route forms D in its dQ kernel
  if (attn_bwd_tc_supported(std::is_same<T, bf16>::value ? NT_BF16 : NT_F32, D) && p.T_q > 0 && p.T_k > 0 &&
      p.B > 0)
    return launch_attn_bwd_tc(p, Dbuf, status, s);
  if (wq > 0)
    rowdot_kernel<T, D><<<(unsigned)((p.T_q + 7) / 8), 256, 0, s>>>((const T*)p.o, (const T*)p.d_o, p.T_q, p.H,
                                                                    Dbuf);
  if (wq > 0) {
    dq_kernel<T, D><<<gq, kWarps * 32, 0, s>>>((const T*)p.q, (const T*)p.k, (const T*)p.v, (const T*)p.d_o, p.lse,
                                             Dbuf, p.cu_q, p.cu_k, p.B, p.T_q, p.T_k, p.H, p.scale, p.causal,
                                             (T*)p.dq, status);
  }
  if (wk > 0)
    dkv_kernel<T, D><<<gk, kWarps * 32, 0, s>>>((const T*)p.q, (const T*)p.k, (const T*)p.v, (const T*)p.d_o, p.lse,
                                              Dbuf, p.cu_q, p.cu_k, p.B, p.T_q, p.T_k, p.H, p.scale, p.causal,
                                              (T*)p.dk, (T*)p.dv, status);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const AttnBwdProblem& p, float* Dbuf, unsigned int* status, cudaStream_t s) {
  switch (p.d) {
    case 32: return launch_d<T, 32>(p, Dbuf, status, s);
    case 64: return launch_d<T, 64>(p, Dbuf, status, s);
    case 128: return launch_d<T, 128>(p, Dbuf, status, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool attn_bwd_supported(int d) { return d == 32 || d == 64 || d == 128; }

cudaError_t launch_attn_bwd(nt_dtype dt, const AttnBwdProblem& p, float* Dbuf, unsigned int* status,
                            cudaStream_t s) {
  return dt == NT_BF16 ? launch_t<bf16>(p, Dbuf, status, s) : launch_t<float>(p, Dbuf, status, s);
}

}  // namespace nt
