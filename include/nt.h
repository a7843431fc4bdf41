/*
 * nt.h -- C ABI of libnt: the packed multi-ragged single->pair->single block
 * and variable-length (cu_seqlens) attention, for NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations:
 *   [DL]  "DanLing NestedTensor: Composable Multi-Ragged Tensors for Deep
 *         Learning" -- section 3 Eq. 1 (the block), section 3.1 Eq. 2 and
 *         Figure 2 (packed storage, offsets, row splits), section 3.2 Eq. 3
 *         (packed row of ragged coordinates) and Eq. 4 (reduction consuming a
 *         pair axis), section 3.3 (dense work on packed rows; projections are
 *         V W^T + b), Appendix A (structural invariants).
 *   [VA]  "Variable-length attention and data packing" -- sections "What it
 *         is", "How it works" and "Core math" (C) (attention restricted to
 *         each cu_seqlens segment, block-diagonal mask).
 *
 * Conventions shared by every call
 *   - Ownership: the caller owns every buffer and the stream.  The library
 *     never allocates or frees device memory.  Pointers named d_* and every
 *     tensor argument are DEVICE pointers; nt_partition lives in HOST memory.
 *   - Layout: row-major, features innermost.  Weights are (out, in) so that
 *     y = x W^T + b ([DL] section 3.3).  Packed singles are (T, C_s); packed
 *     pair cells are (P, C_z) with cell (a, b) of sample i at row
 *     pair_off[i] + a * N_i + b ([DL] Eq. 3).
 *   - dtype: NT_BF16 -- activations and weights bf16, LayerNorm parameters and
 *     biases fp32, all accumulation fp32.  NT_F32 -- every operand fp32.
 *   - Alignment: every pointer 16-byte aligned; feature widths multiples of
 *     8 (bf16) or 4 (fp32).  Otherwise NT_ERR_INVALID / NT_ERR_UNSUPPORTED.
 *   - Empty batches: an array with no elements (the singles, m or s_out of a
 *     batch with T = 0, the pair state of one with P = 0, a workspace of 0
 *     bytes) may be passed as NULL; weights and parameters may not.  Such a
 *     call writes what it has (e.g. zero parameter gradients, a loss of 0).
 *   - Asynchrony: calls enqueue work on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and return.  nt_partition_build (and its
 *     _rect and _with_rows forms) is the one call that synchronises the
 *     stream, once, to return the totals.  The partition kernel writes them
 *     straight into a 64-byte mapped pinned host buffer per calling thread
 *     (allocated on first use, kept for the life of the process), so no copy
 *     engine is involved and the read-back does not queue behind large
 *     device-to-host copies on other streams.  The library allocates no
 *     device memory.
 *   - Errors: argument errors are detected on the host before anything is
 *     enqueued; the call then writes nothing.  NT_ERR_CUDA reports a launch
 *     failure (outputs undefined).  Device-side checks (bounded waits, data
 *     checks) set a device status word that nt_device_status() reads.
 *     nt_last_error() gives a one-line detail of the last failure on the
 *     calling thread.
 */
#ifndef NT_H_
#define NT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NT_OK = 0,
  NT_ERR_INVALID = 1,      /* bad argument: null, negative, misaligned, mismatched */
  NT_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels implement */
  NT_ERR_OVERFLOW = 3,     /* a total does not fit its index type */
  NT_ERR_CUDA = 4,         /* CUDA runtime/launch error */
  NT_ERR_TIMEOUT = 5,      /* a bounded device-side wait ran out */
  NT_ERR_DEVICE_CHECK = 6  /* a device-side data check failed */
} nt_status;

typedef enum { NT_F32 = 0, NT_BF16 = 1 } nt_dtype;

/*
 * Partitions of a packed batch of B samples with lengths N_i ([DL] section
 * 3.1, Figure 2; Appendix A "Structural invariants").
 *   cu_seqlens[B+1]  sample offsets of the singles, o_i = sum_{k<i} N_k
 *                    (= eta_i of Eq. 4); int32 (the cu_seqlens convention).
 *   pair_off[B+1]    sample offsets of the square pairs, sum_{k<i} N_k^2.
 *   row_start[T+1]   second-level splits: first cell of every pair row,
 *                    row_start[cu_seqlens[i] + a] = pair_off[i] + a * N_i,
 *                    row_start[T] = P.
 *   row_sample[T]    sample index owning each single row / pair row.
 * T = sum N_i, P = sum N_i^2, max_len = max N_i.  All pointers are device
 * pointers owned by the caller; the struct itself is host memory.
 *
 * Rectangular pair states ([DL] section 3.2 "Consuming one logical axis",
 * Eq. 4): sample i has N_i rows and M_i columns, its cells are packed at
 * pair_off[i] + a * M_i + b with pair_off the exclusive scan of N_i * M_i,
 * and row_start[cu_seqlens[i] + a] = pair_off[i] + a * M_i.  The column
 * fields below describe M_i; nt_partition_build sets them to alias the row
 * fields (M_i = N_i), and a struct whose col_lengths is NULL is read as
 * square too.  T, max_len, lengths and cu_seqlens always describe the rows.
 */
typedef struct nt_partition {
  int32_t B;
  int64_t T;
  int64_t P;
  int32_t max_len;
  const int32_t* lengths;
  const int32_t* cu_seqlens;
  const int64_t* pair_off;
  const int64_t* row_start;   /* NULL until nt_partition_rows */
  const int32_t* row_sample;  /* NULL until nt_partition_rows */
  const int32_t* col_lengths;     /* M_i [B], or NULL for square pairs */
  const int32_t* col_cu_seqlens;  /* [B+1] exclusive scan of M_i (column singles) */
  int64_t T_cols;                 /* sum M_i */
  int32_t max_col_len;            /* max M_i */
} nt_partition;

/*
 * nt_partition_build -- exact sizes to tensor-backed offsets ([DL] Eq. 2,
 * Figure 2, Appendix A): exclusive scans of N_i and of N_i^2 on the device.
 *   d_lengths     [B] int32, N_i >= 0 (zero-length samples allowed).
 *   B             number of samples, >= 0 (an empty batch gives T = P = 0).
 *   d_cu_seqlens  [B+1] int32 out.   d_pair_off [B+1] int64 out.
 *   d_totals      [4] int64 device scratch: T, P, max_len, check word.
 *   out           host struct filled with B, T, P, max_len and the pointers;
 *                 row_start / row_sample are set to NULL.
 * Synchronises `stream` once to read the totals.  Returns NT_ERR_INVALID if
 * some N_i < 0 and NT_ERR_OVERFLOW if T does not fit int32 (out->T, out->P
 * are still filled).  Integer-exact.
 */
nt_status nt_partition_build(const int32_t* d_lengths, int32_t B, int32_t* d_cu_seqlens,
                             int64_t* d_pair_off, int64_t* d_totals, nt_partition* out,
                             void* stream);

/*
 * nt_partition_build_rect -- partitions of rectangular pair states ([DL]
 * section 3.2 "Consuming one logical axis", Eq. 4; Appendix A.1, the
 * rectangular variant with distinct row and column inputs).
 *   d_rows, d_cols  [B] int32, N_i >= 0 rows and M_i >= 0 columns.
 *   d_cu_rows       [B+1] int32 out, exclusive scan of N_i (eta of Eq. 4).
 *   d_cu_cols       [B+1] int32 out, exclusive scan of M_i.
 *   d_pair_off      [B+1] int64 out, exclusive scan of N_i * M_i.
 *   d_totals        [8] int64 device scratch.
 *   out             filled like nt_partition_build, with the column fields
 *                   pointing at d_cols / d_cu_cols.
 * Synchronises `stream` once.  NT_ERR_INVALID for a negative length,
 * NT_ERR_OVERFLOW if sum N_i or sum M_i does not fit int32.  Integer-exact.
 */
nt_status nt_partition_build_rect(const int32_t* d_rows, const int32_t* d_cols, int32_t B,
                                  int32_t* d_cu_rows, int32_t* d_cu_cols, int64_t* d_pair_off,
                                  int64_t* d_totals, nt_partition* out, void* stream);

/*
 * nt_partition_rows -- second-level row splits of the pair state ([DL]
 * Figure 2: 1 + sum N_i entries; Eq. 3 with b = 0; rows of a rectangular
 * state are M_i cells long, Eq. 4).
 *   part          a partition from nt_partition_build (T, P known).
 *   d_row_start   [T+1] int64 out.   d_row_sample [T] int32 out.
 * Sets part->row_start and part->row_sample.  Asynchronous.
 */
nt_status nt_partition_rows(nt_partition* part, int64_t* d_row_start, int32_t* d_row_sample,
                            void* stream);

/*
 * nt_partition_build_with_rows -- nt_partition_build and nt_partition_rows
 * in one call and one host round trip: the row-split kernel follows the scan
 * in the stream and reads T and P from d_totals, so only the totals come
 * back to the host.  For 1 <= B <= 1024 and T_cap <= 65,536 the scan and the
 * row splits run as one single-CTA launch (same outputs).  For callers that
 * know an upper bound on T, such as the row count of the packed singles they
 * hold.
 *   T_cap          >= 0; d_row_start holds T_cap + 1 entries and d_row_sample
 *                  max(T_cap, 1).  Device writes never go past them.
 *   other arguments as in nt_partition_build / nt_partition_rows; on NT_OK
 *                  *out is filled including row_start and row_sample.
 * Returns NT_ERR_INVALID if the lengths sum to more than T_cap (the row
 * splits are then incomplete; *out still holds the totals), and the errors
 * of nt_partition_build.  Synchronises `stream` once.
 */
nt_status nt_partition_build_with_rows(const int32_t* d_lengths, int32_t B, int64_t T_cap,
                                       int32_t* d_cu_seqlens, int64_t* d_pair_off, int64_t* d_totals,
                                       int64_t* d_row_start, int32_t* d_row_sample,
                                       nt_partition* out, void* stream);

/* Bytes of device workspace nt_pair_broadcast needs for a square partition:
 * the two projected single representations u and v in fp32, 2 * T * C_z * 4. */
size_t nt_pair_broadcast_workspace_bytes(int64_t T, int32_t C_z);

/* The same for a rectangular partition: (T_rows + T_cols) * C_z * 4. */
size_t nt_pair_broadcast_workspace_bytes_rect(int64_t T_rows, int64_t T_cols, int32_t C_z);

/*
 * nt_pair_broadcast -- pair construction of [DL] Eq. 1, first line, with the
 * broadcast of section 3.2 "Creating axes through broadcasting":
 *     u = s_left W_a^T,  v = s_right W_b^T            (fp32)
 *     z[pair_off[i] + a M_i + b, :] = u[cu_i + a] + v[col_cu_i + b]
 * over the P = sum N_i M_i cells only (M_i = N_i and col_cu = cu for square
 * pairs); no activation at construction ([DL] Appendix A.1).
 *   part          partition with row splits (nt_partition_rows done).
 *   s_left        [T, C_s] row singles.
 *   s_right       [T_cols, C_s] column singles (the same pointer as s_left
 *                 for square pairs built from one single representation).
 *   W_a, W_b      [C_z, C_s].        z [P, C_z] out.
 *   workspace     >= (T + T_cols) * C_z * 4 device bytes (see the two
 *                 workspace-size calls), 16-byte aligned; holds u and v
 *                 while the call runs.
 * Asynchronous.  Rounds z once to the I/O dtype (round-to-nearest-even).
 */
nt_status nt_pair_broadcast(const nt_partition* part, nt_dtype dtype, const void* s_left,
                            const void* s_right, int32_t C_s, const void* W_a, const void* W_b,
                            int32_t C_z, void* z, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * nt_pair_broadcast_noalloc -- nt_pair_broadcast for callers that cannot
 * allocate device memory.  The pages describe no counterpart: it is a
 * property of this library, not of the method.
 *
 * nt_pair_broadcast needs a caller workspace for u and v.  Some callers
 * cannot provide one: a plug-in whose host framework owns every device
 * allocation and hands it none, or a real-time loop that must not pay for
 * (or risk failing) an allocation on its hot path.  This call takes the same
 * arguments minus the workspace and keeps u and v in a fixed array that the
 * library declares in device memory (8 MiB, held on every GPU that loads the
 * library until the process exits).  It allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *   Limit: (T + T_cols) * C_z <= 2,097,152 (2 * T * C_z for square
 *   partitions); larger problems return
 *   NT_ERR_UNSUPPORTED (see nt_last_error) and enqueue nothing.
 *   Set-up: every call looks up the array's device address
 *   (cudaGetSymbolAddress) with the calling thread's device current, so the
 *   call stays valid across cudaDeviceReset.  With CUDA's default lazy
 *   module loading, the first call on a device is what loads the array onto
 *   that device: that call commits its 8 MiB of device memory and is where
 *   an out-of-memory failure would appear (as NT_ERR_CUDA; with
 *   CUDA_MODULE_LOADING=EAGER the array is committed when the library loads
 *   instead).  A caller that must not allocate on its hot path makes one
 *   warm-up call on each device outside it; make that first call before any
 *   stream capture on the device.
 *   Sharing: every call uses the same array.  Calls that overlap on the GPU
 *   (other streams, other host threads on the same device) race on it; order
 *   them on one stream.  The kernels overwrite every element of u and v they
 *   read, so earlier contents never reach a result and nothing needs clearing.
 * Other arguments, outputs and errors are those of nt_pair_broadcast.
 */
nt_status nt_pair_broadcast_noalloc(const nt_partition* part, nt_dtype dtype, const void* s_left,
                                    const void* s_right, int32_t C_s, const void* W_a,
                                    const void* W_b, int32_t C_z, void* z, void* stream);

/*
 * nt_pair_transition -- residual feature update of [DL] Eq. 1, second line,
 * on every packed cell (section 3.2 "Retaining structure through feature
 * transformations"; section 3.3 "Dense work across valid positions"):
 *     x  = LN(z) = (z - mean) / sqrt(var + ln_eps) * ln_gamma + ln_beta
 *     z~ = z + W2 ReLU(W1 x + b1) + b2
 * LayerNorm over the C_z features of one cell, biased variance.
 *   z_in, z_out   [P, C_z]; z_out may equal z_in (in place).
 *   ln_gamma, ln_beta [C_z] fp32.  W1 [H_t, C_z].  b1 [H_t] fp32 or NULL.
 *   W2 [C_z, H_t].  b2 [C_z] fp32 or NULL.
 * bf16 with C_z = 128 and H_t a multiple of 128 runs on the tcgen05 tensor
 * cores (hidden activations rounded to bf16 before the second GEMM); other
 * shapes and NT_F32 run on fp32 CUDA cores.  Asynchronous.  At most
 * 2^31 - 1025 cells per call (cell rows are 32-bit copy coordinates), else
 * NT_ERR_OVERFLOW; the same bound holds for nt_pair_block_fused.
 */
nt_status nt_pair_transition(const nt_partition* part, nt_dtype dtype, const void* z_in,
                             void* z_out, int32_t C_z, int32_t H_t, const float* ln_gamma,
                             const float* ln_beta, float ln_eps, const void* W1,
                             const float* b1, const void* W2, const float* b2, void* stream);

/*
 * nt_pair_transition_swiglu -- the transition with the SwiGLU update that
 * [DL] measures (Eq. 1: h is "a SwiGLU feature update"; Appendix A.1:
 * transition expansion four):
 *     y  = LN(z)                                      (as nt_pair_transition)
 *     z~ = z + W2 (SiLU(W1 y + b1) * (W3 y + b3)) + b2,  SiLU(x) = x sigmoid(x)
 *   W1 [H_t, C_z] the gate projection, W3 [H_t, C_z] the value projection,
 *   W2 [C_z, H_t]; b1, b3 [H_t] and b2 [C_z] fp32 or NULL.
 * bf16 with C_z = 128 and H_t a multiple of 64 runs on the tensor cores
 * (hidden chunks of 64 units, gate and value from one MMA); other shapes
 * and NT_F32 on CUDA cores.  W3 == NULL is NT_ERR_INVALID.  Other
 * arguments, errors and in-place use are those of nt_pair_transition.
 */
nt_status nt_pair_transition_swiglu(const nt_partition* part, nt_dtype dtype, const void* z_in,
                                    void* z_out, int32_t C_z, int32_t H_t, const float* ln_gamma,
                                    const float* ln_beta, float ln_eps, const void* W1,
                                    const float* b1, const void* W3, const float* b3,
                                    const void* W2, const float* b2, void* stream);

/*
 * nt_pair_transition_cells -- the transition of nt_pair_transition (W3 NULL)
 * or nt_pair_transition_swiglu (W3 given) over n_cells consecutive packed
 * cells, with no partition: the transition maps every cell's feature vector
 * on its own ("DanLing NestedTensor" section 3.3, dense work across valid
 * positions), so a caller may run it over any slice [c0, c0 + n_cells) of a
 * pair state by passing z_in + c0 * C_z and z_out + c0 * C_z, for instance to
 * read finished slices back while the next one is computed.  Every cell's
 * result is bit-identical to the whole-state call's.
 *   n_cells        >= 0 (0 is a no-op, whatever the pointers).
 *   other arguments as in nt_pair_transition / nt_pair_transition_swiglu
 *                  (b3 is ignored when W3 is NULL).
 * Asynchronous; errors as for nt_pair_transition.
 */
nt_status nt_pair_transition_cells(int64_t n_cells, nt_dtype dtype, const void* z_in, void* z_out,
                                   int32_t C_z, int32_t H_t, const float* ln_gamma,
                                   const float* ln_beta, float ln_eps, const void* W1,
                                   const float* b1, const void* W3, const float* b3,
                                   const void* W2, const float* b2, void* stream);

/*
 * nt_pair_reduce -- the column mean of [DL] Eq. 1, third line, as the
 * segmented sum of Eq. 4 divided by the row length M_i (= N_i for square
 * pairs; [DL] Appendix A.1 for the rectangular variant):
 *     m[cu_i + a, :] = (1/M_i) sum_b z[pair_off[i] + a M_i + b, :]
 * (zero for a sample with M_i = 0, whose column sum is empty)
 * then, if W_g is not NULL:  s_out = s_in + m W_g^T + b_g.
 *   z [P, C_z].  m [T, C_z] out (fp32 accumulation, stored in the I/O dtype).
 *   W_g [C_s, C_z] or NULL.  b_g [C_s] fp32 or NULL.  s_in [T, C_s] or NULL
 *   (no residual).  s_out [T, C_s] out (required when W_g is given; may
 *   equal s_in).
 * Asynchronous.
 */
nt_status nt_pair_reduce(const nt_partition* part, nt_dtype dtype, const void* z, int32_t C_z,
                         void* m, const void* W_g, const float* b_g, const void* s_in,
                         void* s_out, int32_t C_s, void* stream);

/* Bytes of device workspace nt_pair_block_fused needs: u (T x C_z), v
 * (T_cols x C_z) and the fp32 row sums (T x C_z), (2 T + T_cols) * C_z * 4. */
size_t nt_pair_block_fused_workspace_bytes(int64_t T, int64_t T_cols, int32_t C_z);

/*
 * nt_pair_block_fused -- the whole single -> pair -> single block of [DL]
 * Eq. 1 in one pass over the pair state: the broadcast is computed inside
 * the transition's prologue and the row sums of Eq. 4 inside its epilogue,
 * so z is never written to HBM and z~ is written once (256 bytes per cell in
 * bf16 instead of the 1,024 of the three separate calls).
 *     u = s_left W_a^T, v = s_right W_b^T
 *     z~[cell (a, b) of sample i] = transition(u[cu_i + a] + v[col_cu_i + b])
 *     m = column mean of z~ (divided by M_i);  s_out = s_left + m W_g^T + b_g
 * The transition is the ReLU one (W3 == NULL) or the SwiGLU one (W3 given),
 * with the arguments of nt_pair_transition / nt_pair_transition_swiglu.
 *   part      partition with row splits; square or rectangular.
 *   z_out     [P, C_z] out: z~ (the pair state the block returns).
 *   m         [T, C_z] out.   s_out [T, C_s] out when W_g is given.
 *   workspace >= nt_pair_block_fused_workspace_bytes(T, T_cols, C_z) bytes,
 *             16-byte aligned.
 * z~ equals what the three calls produce bit for bit (same roundings: z is
 * rounded to bf16 before the LayerNorm and the residual); m differs only in
 * the order of the fp32 row sums.  bf16 with C_z = 128 runs fused on the
 * tensor cores; other shapes run the three calls' kernels in sequence.
 * Asynchronous; errors as for the three calls.
 */
nt_status nt_pair_block_fused(const nt_partition* part, nt_dtype dtype, const void* s_left,
                              const void* s_right, int32_t C_s, const void* W_a, const void* W_b,
                              int32_t C_z, int32_t H_t, const float* ln_gamma, const float* ln_beta,
                              float ln_eps, const void* W1, const float* b1, const void* W3,
                              const float* b3, const void* W2, const float* b2, const void* W_g,
                              const float* b_g, void* z_out, void* m, void* s_out, void* workspace,
                              size_t workspace_bytes, void* stream);

/* Bytes of device workspace nt_pair_reduce_loss needs (a constant: the
 * loss's partial sums and up to 8,192 per-CTA partials of the pair term). */
size_t nt_pair_reduce_loss_workspace_bytes(void);

/*
 * nt_pair_reduce_loss -- nt_pair_reduce with the g projection, and the Eq. 5
 * loss of [DL] Appendix A.1 on the block's two outputs (s_out and z), in one
 * call that reads z once: the reduce's pass over the cells also sums each
 * pair row's squares, weighted by beta_i of its sample, into per-CTA
 * partials; the single-row term follows over s_out, and one block adds both
 * in a fixed order (the result does not depend on scheduling, only on the
 * device's SM count, which sets the reduce's grid).  The same loss as
 * nt_pair_block_loss up to the order of its sums.
 *   z, C_z, m, W_g (required), b_g, s_in, s_out, C_s  as for nt_pair_reduce.
 *   d_loss     one fp32 on the device, written.
 *   workspace  >= nt_pair_reduce_loss_workspace_bytes(), 16-byte aligned.
 * C_z not a multiple of 8 (fp32): the loss reads z again (nt_pair_block_loss's
 * path).  Errors as for nt_pair_reduce, plus NT_ERR_INVALID for a NULL W_g,
 * d_loss or workspace, a NULL z when P > 0 or a NULL m or s_out when T > 0
 * (an empty batch writes a zero loss).  Asynchronous.
 */
nt_status nt_pair_reduce_loss(const nt_partition* part, nt_dtype dtype, const void* z, int32_t C_z, void* m,
                              const void* W_g, const float* b_g, const void* s_in, void* s_out, int32_t C_s,
                              float* d_loss, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace nt_pair_block_loss needs (its partial sums). */
size_t nt_pair_block_loss_workspace_bytes(void);

/*
 * nt_pair_block_loss -- the sample-weighted squared loss of [DL] Appendix
 * A.1, Eq. 5, on both outputs of one block (square pairs, the packed layout
 * being a leading one, S = 1):
 *     L = sum_i alpha_i ||X~_i||_F^2 / (C_s sum_i N_i)
 *       + sum_i beta_i  ||P~_i||_F^2 / (C_z sum_i N_i^2),
 *     alpha_i = 1 + i / B,  beta_i = 1.5 - i / (2 B),
 * with X~_i the sample's rows of s_out and P~_i its cells of z_tilde.
 *   s_out     [T, C_s], z_tilde [P, C_z] in the I/O dtype.
 *   d_loss    one fp32 on the device, written.  The squared sums accumulate
 *             in fp32 per thread and in double across the batch, in a fixed
 *             order (the result does not depend on scheduling).
 *   ds_out    [T, C_s] fp32 or NULL: if given, dL/ds_out = 2 alpha_i X~ / (C_s T).
 *   dz_tilde  [P, C_z] fp32 or NULL: if given, dL/dz~ = 2 beta_i P~ / (C_z P).
 *   workspace >= nt_pair_block_loss_workspace_bytes(), 16-byte aligned.
 * Asynchronous.  Errors as for nt_pair_reduce.
 */
nt_status nt_pair_block_loss(const nt_partition* part, nt_dtype dtype, const void* s_out, int32_t C_s,
                             const void* z_tilde, int32_t C_z, float* d_loss, float* ds_out, float* dz_tilde,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace nt_pair_block_backward needs for this dtype and
 * these sizes: u, v, dM, du, dv ([T, C_z] fp32 each) and dz ([P, C_z] fp32),
 * (5 T + P) * C_z * 4 rounded up to 256; for bf16 with C_z = 128 and H_t a
 * multiple of 128 (the tensor-core route), also the cells' rows LN(z) and
 * dP~ ([P, C_z] bf16 each), H and dA ([P, H_t] bf16 each), the LayerNorm
 * statistics ([P, 2] fp32), the transposed W1 and W2 and the split
 * weight-gradient partials.  0 for negative sizes. */
size_t nt_pair_block_backward_workspace_bytes(nt_dtype dtype, int64_t T, int64_t P, int32_t C_z, int32_t H_t);

/*
 * nt_pair_block_backward -- gradients of one single -> pair -> single block
 * ([DL] Eq. 1 with the ReLU transition of nt_pair_transition) with respect to
 * its singles and every parameter, for upstream gradients of its two
 * outputs (for Eq. 5, the ds_out and dz_tilde that nt_pair_block_loss
 * writes).  The chain rule of Eq. 1 ([DL] section 3.4: gradients flow from
 * the eager loss back through the pair update, the reduction and the
 * projections):
 *     dM = ds_out W_g,  dW_g = ds_out^T m,  db_g = sum ds_out
 *     dP~ = dz_tilde + dM[row] / N_i            (the column mean's backward)
 *     A = LN(z) W1^T + b1:  dH = dP~ W2,  dA = dH [A > 0],  dY = dA W1,
 *       dW1 = dA^T LN(z),  dW2 = dP~^T ReLU(A),  db1 = sum dA,  db2 = sum dP~
 *     dz = dP~ + the LayerNorm backward of dY   (dgamma, dbeta)
 *     du = row sums of dz,  dv = column sums of dz (within each sample)
 *     dW_a = du^T s,  dW_b = dv^T s,  ds = ds_out + du W_a + dv W_b
 * z is rebuilt from s (u = s W_a^T, v = s W_b^T, rounded to the I/O dtype as
 * the forward rounds it), so the forward's pair state need not be kept.
 *   part       square partition with row splits (rectangular ones are
 *              NT_ERR_UNSUPPORTED).
 *   s          [T, C_s] the block's input singles;  m [T, C_z] the row means
 *              the forward's nt_pair_reduce wrote.
 *   W_a, W_b, ln_gamma, ln_beta, ln_eps, W1, b1 (nullable), W2, W_g: the
 *              forward's parameters (b2 and b_g do not enter the gradients).
 *   ds_out     [T, C_s] fp32, required;  dz_tilde [P, C_z] fp32 or NULL (no
 *              gradient reaches z~ from downstream).
 *   ds         [T, C_s] fp32 out.  dW_a, dW_b [C_z, C_s], dgamma, dbeta [C_z],
 *              dW1 [H_t, C_z], db1 [H_t], dW2 [C_z, H_t], db2 [C_z],
 *              dW_g [C_s, C_z], db_g [C_s]: fp32 out, overwritten (the call
 *              clears them on its stream before accumulating).
 *   workspace  >= nt_pair_block_backward_workspace_bytes(dtype, T, P, C_z,
 *              H_t) bytes.
 * Supported: 8 <= C_z <= 128, H_t a multiple of 64, either dtype.  bf16 with
 * C_z = 128 and H_t a multiple of 128 runs the pair cells on the tcgen05
 * tensor cores: LN(z) and dP~ as bf16 rows, H = ReLU(LN(z) W1^T + b1),
 * dA = (dP~ W2) where H > 0 and dY = dA W1 as GEMMs, dW1 = dA^T LN(z) and
 * dW2 = dP~^T H (with db1, db2) split over the cells and summed in a fixed
 * order; the GEMM operands are bf16, every accumulation fp32.  Otherwise
 * CUDA cores in fp32.  dgamma, dbeta and the single-row gradients
 * accumulate with fp32 atomics, so they are not bit-reproducible from run
 * to run.  Asynchronous.
 */
nt_status nt_pair_block_backward(const nt_partition* part, nt_dtype dtype, const void* s, int32_t C_s,
                                 const void* W_a, const void* W_b, int32_t C_z, int32_t H_t, const float* ln_gamma,
                                 const float* ln_beta, float ln_eps, const void* W1, const float* b1, const void* W2,
                                 const void* W_g, const void* m, const float* ds_out, const float* dz_tilde,
                                 float* ds, float* dW_a, float* dW_b, float* dgamma, float* dbeta, float* dW1,
                                 float* db1, float* dW2, float* db2, float* dW_g, float* db_g, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* Bytes of device workspace nt_pair_block_loss_backward needs: the loss's
 * partial sums, dL/dX~ ([T, C_s] fp32), dL/dz~ ([P, C_z] fp32) except on the
 * tensor-core route, and nt_pair_block_backward_workspace_bytes(dtype, T, P,
 * C_z, H_t), each part rounded up to 256 bytes.  0 for negative sizes. */
size_t nt_pair_block_loss_backward_workspace_bytes(nt_dtype dtype, int64_t T, int64_t P, int32_t C_s,
                                                   int32_t C_z, int32_t H_t);

/*
 * nt_pair_block_loss_backward -- the Eq. 5 loss of [DL] Appendix A.1 on the
 * block's outputs and the block's gradients for it, in one call: the same
 * loss as nt_pair_block_loss and the same gradients as nt_pair_block_backward
 * given that call's ds_out and dz_tilde, value for value (the upstream
 * gradients are formed by the same fp32 operations).  dL/dz~ = gp_i P~ with
 * gp_i = 2 beta_i / (C_z sum_i N_i^2) is linear in z~, so on the tensor-core
 * route (bf16, C_z = 128, H_t a multiple of 128) it is never stored: the
 * two kernels that read it form it from z~ ([P, C_z] bf16, half the bytes of
 * the fp32 gradient, and no pass that writes it).  Other routes store it in
 * the workspace first.
 *   s_out, z_tilde   the block's outputs (as nt_pair_block_loss takes them).
 *   d_loss           one fp32 on the device, written.
 *   every other argument as for nt_pair_block_backward (no ds_out or
 *   dz_tilde: they are this loss's).
 *   workspace  >= nt_pair_block_loss_backward_workspace_bytes(dtype, T, P,
 *              C_s, C_z, H_t) bytes, 16-byte aligned.
 * Errors as for nt_pair_block_backward, plus NT_ERR_INVALID for a NULL
 * d_loss, s_out (T > 0) or z_tilde (P > 0).  Asynchronous.
 */
nt_status nt_pair_block_loss_backward(const nt_partition* part, nt_dtype dtype, const void* s, int32_t C_s,
                                      const void* W_a, const void* W_b, int32_t C_z, int32_t H_t,
                                      const float* ln_gamma, const float* ln_beta, float ln_eps, const void* W1,
                                      const float* b1, const void* W2, const void* W_g, const void* m,
                                      const void* s_out, const void* z_tilde, float* d_loss, float* ds, float* dW_a,
                                      float* dW_b, float* dgamma, float* dbeta, float* dW1, float* db1, float* dW2,
                                      float* db2, float* dW_g, float* db_g, void* workspace, size_t workspace_bytes,
                                      void* stream);

/*
 * nt_varlen_attn_workspace_bytes -- bytes of device workspace that
 * nt_varlen_attn and nt_varlen_attn_qk take for their work counter (a small
 * constant, 256).  The counter belongs to the call that is given it: calls
 * that may overlap on the GPU (other streams, other host threads, replays of
 * a captured graph on several streams) each need a workspace of their own;
 * calls ordered on one stream may share one.  Each call clears its counter
 * on its own stream before the kernel runs, so nothing needs clearing by the
 * caller, and the library keeps no mutable device state between calls.
 */
size_t nt_varlen_attn_workspace_bytes(void);

/*
 * nt_varlen_attn -- softmax attention restricted to each cu_seqlens segment
 * ([VA] "What it is", "How it works"; [DL] section 3.3 "Attention through
 * packed blocks"): for token t of segment i and head h,
 *     O[t, h, :] = sum_{k in [cu_i, cu_{i+1})} softmax_k(scale q_t.k_k) v_k
 * non-causal; equivalent to the block-diagonal mask seg(t) == seg(k) of
 * [VA] "Core math" (C) with no padded rectangle formed.
 *   q, k, v, o    [T, H, d] token-major, contiguous.
 *   d_cu_seqlens  [B+1] int32, non-decreasing, cu[0] = 0, cu[B] = T.
 *   max_len       max segment length (>= every cu[i+1] - cu[i]).
 *   scale         score scale, finite and > 0 (d^-1/2 for the usual
 *                 attention); anything else is NT_ERR_INVALID.
 *   lse           [H, T] fp32 natural-log log-sum-exp, or NULL.
 *   workspace     >= nt_varlen_attn_workspace_bytes() device bytes, 16-byte
 *                 aligned, or NULL (with workspace_bytes 0).  With a
 *                 workspace, batches of short segments (mean length up to
 *                 768) run on persistent CTAs that take work items from a
 *                 counter kept there; without one, every batch runs one CTA
 *                 per (segment, query tile, head), which needs no shared
 *                 state but pays a per-item start-up cost.  Same results
 *                 either way.
 * bf16 with d = 64 runs on the tcgen05 tensor cores; NT_F32 and other head
 * widths (32, 64, 128) run on fp32 CUDA cores.  Asynchronous.  Identical to
 * nt_varlen_attn_qk with d_cu_seqlens_k = d_cu_seqlens, T_k = T, causal = 0.
 */
nt_status nt_varlen_attn(nt_dtype dtype, const void* q, const void* k, const void* v,
                         const int32_t* d_cu_seqlens, int32_t B, int64_t T, int32_t max_len,
                         int32_t H, int32_t d, float scale, void* o, float* lse, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * nt_varlen_attn_qk -- varlen attention with separate query and key
 * segments, and an optional causal mask.  Query segment b,
 * [cu_q[b], cu_q[b+1]), attends to key segment b, [cu_k[b], cu_k[b+1]); the
 * output adopts the query structure ([DL] section 3.3 "Attention through
 * packed blocks": attention over packed blocks, query and key lengths may
 * differ).  With causal = 1, query i of a segment with n_q queries and n_k
 * keys sees the keys j <= i + (n_k - n_q) (the diagonal aligned to the
 * bottom-right corner; for self-attention, j <= i).  [VA] "How to use it":
 * the varlen call of the page's template sets the causal flag.  A query that sees no key
 * (n_k = 0, or causal with i + n_k - n_q < 0) gets O = 0 and lse = -inf.
 *   q, o          [T_q, H, d] token-major, contiguous.
 *   k, v          [T_k, H, d] token-major, contiguous (may be NULL if T_k = 0).
 *   d_cu_seqlens_q, d_cu_seqlens_k
 *                 [B+1] int32 each, non-decreasing, starting at 0, ending at
 *                 T_q and T_k.  Offsets inconsistent with T_q / T_k are caught
 *                 on the device: nothing is written for those segments and
 *                 nt_device_status reports NT_ERR_DEVICE_CHECK.
 *   max_len_q     max query segment length (>= every cu_q[b+1] - cu_q[b]).
 *   scale         finite and > 0.
 *   causal        0 or 1.
 *   lse           [H, T_q] fp32 natural-log log-sum-exp, or NULL.
 *   workspace, workspace_bytes  as in nt_varlen_attn.
 * Host errors: NT_ERR_INVALID (bad sizes, flags, scale, NULL or misaligned
 * pointers, a workspace smaller than nt_varlen_attn_workspace_bytes()),
 * NT_ERR_OVERFLOW (T_q or T_k beyond int32), NT_ERR_UNSUPPORTED (head
 * width).  bf16 with d = 64 and T_k > 0 runs on the tensor cores; the rest
 * on CUDA cores.  Asynchronous on `stream`; buffers stay owned by the
 * caller.
 */
nt_status nt_varlen_attn_qk(nt_dtype dtype, const void* q, const void* k, const void* v,
                            const int32_t* d_cu_seqlens_q, const int32_t* d_cu_seqlens_k, int32_t B,
                            int64_t T_q, int64_t T_k, int32_t max_len_q, int32_t H, int32_t d, float scale,
                            int32_t causal, void* o, float* lse, void* workspace, size_t workspace_bytes,
                            void* stream);

/* Bytes of device workspace nt_varlen_attn_bwd needs: the H * T_q fp32 row
 * sums rowsum(dO * O), rounded up to 256 bytes, then 256 bytes for the work
 * counters of its persistent kernels (cleared by the call on its stream).
 * Overlapping backward calls need workspaces of their own. */
size_t nt_varlen_attn_bwd_workspace_bytes(int64_t T_q, int32_t H);

/*
 * nt_varlen_attn_bwd -- gradients of nt_varlen_attn_qk (and so of
 * nt_varlen_attn) with respect to q, k and v for an upstream gradient d_o
 * (the backward of [VA]'s varlen attention, as training needs it): per
 * segment and head, with P rebuilt from the forward's natural-log lse,
 *     dV = P^T dO,  dS = P * (dO V^T - rowsum(dO * O)),
 *     dQ = scale dS K,  dK = scale dS^T Q
 * (masked entries, causal or across segments, get no gradient; a query that
 * saw no key, lse = -inf, contributes nothing).
 *   q, o, d_o, dq  [T_q, H, d];  k, v, dk, dv [T_k, H, d]; token-major,
 *                  contiguous, dtype as given; dq, dk, dv are overwritten.
 *   lse            [H, T_q] fp32, the forward's (natural log).
 *   d_cu_seqlens_q, d_cu_seqlens_k, scale, causal: as in nt_varlen_attn_qk.
 *   max_len_q, max_len_k  longest query / key segment (>= every
 *                  cu[b+1] - cu[b] of the side); they size the grid of the
 *                  tensor-core path, which flags NT_ERR_DEVICE_CHECK when a
 *                  segment is longer than stated.
 *   workspace      >= nt_varlen_attn_bwd_workspace_bytes(T_q, H) device
 *                  bytes, 16-byte aligned.
 * bf16 with d = 64 runs on the tcgen05 tensor cores (fp32 accumulation in
 * TMEM); d = 32, 64 or 128 in fp32, and bf16 with d = 32 or 128, on CUDA
 * cores (fp32 accumulation).  Asynchronous.  Errors as for
 * nt_varlen_attn_qk; offsets inconsistent with T_q / T_k are caught on the
 * device (NT_ERR_DEVICE_CHECK).
 */
nt_status nt_varlen_attn_bwd(nt_dtype dtype, const void* q, const void* k, const void* v,
                             const void* o, const void* d_o, const float* lse,
                             const int32_t* d_cu_seqlens_q, const int32_t* d_cu_seqlens_k,
                             int32_t B, int64_t T_q, int64_t T_k, int32_t max_len_q,
                             int32_t max_len_k, int32_t H, int32_t d,
                             float scale, int32_t causal, void* dq, void* dk, void* dv,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Synchronises `stream`, then reads and clears the device status word set by
 * device-side checks (bounded waits that ran out: NT_ERR_TIMEOUT; failed data
 * checks: NT_ERR_DEVICE_CHECK).  NT_OK if nothing was flagged. */
nt_status nt_device_status(void* stream);

/* Self-test of the device-side failure reporting; computes nothing.  One
 * CTA waits, through the same bounded mbarrier wait the tensor-core kernels
 * use, on a barrier of its own that
 *   mode 0: another warp completes after about delay_ns: the wait succeeds;
 *   mode 1: nothing completes: the wait runs out after limit_ns, raises the
 *           CTA's abort flag and sets the status word's timeout bit, so the
 *           next nt_device_status returns NT_ERR_TIMEOUT (and clears it);
 *   mode 2: nothing completes, but another warp raises the CTA's abort flag
 *           after delay_ns: the wait gives up early without flagging, as a
 *           CTA's other roles do once one role's wait has run out.
 * d_result: device int64[2], 8-byte aligned, caller-owned; written with
 * [0] = 1 if the wait succeeded, 0 if it gave up, and [1] = the wait's
 * duration in ns.  limit_ns in (0, 2e9], delay_ns at most 2e9, else
 * NT_ERR_INVALID (checked before anything is enqueued).  Asynchronous on
 * `stream`; the CUDA context stays usable in every mode. */
nt_status nt_selftest_bounded_wait(int32_t mode, uint64_t delay_ns, uint64_t limit_ns, int64_t* d_result,
                                   void* stream);

/* Static string naming a status code. */
const char* nt_status_str(nt_status s);

/* One-line detail of the last non-OK status returned on this thread. */
const char* nt_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* NT_H_ */
