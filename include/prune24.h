/*
 * prune24.h -- C ABI of libprune24: 2:4 semi-structured sparse training of
 * transformer FFN layers on one NVIDIA GB300 (sm_103a).
 *
 * What the calls compute (sources: web pages on N:M sparse training, cited by
 * title and section):
 *   - inno4scale "Success story ESPLAG", "Research Topic" / "Solution":
 *     N:M (here 2:4) semi-structured magnitude pruning, a compressed storage
 *     format, a sparse matrix-matrix multiply (SpMM) on sparse tensor cores,
 *     gradual magnitude pruning, and a sparse version of the whole training step.
 *   - NSF PAR award 2340011 listing, SLOPE abstract: the double-pruned backward
 *     pass -- the transposed, already-pruned weight is pruned again with N:M so
 *     that the backward GEMM is sparse as well.
 *   - "To 2:4 Sparsity and Beyond: Neuron-level Activation Function to
 *     Accelerate LLM Pre-Training", abstract: 2:4 weights in every FFN matmul,
 *     with sparse activations on top.
 *   - "Sparser, Faster, Lighter Transformer Language Models", training
 *     strategy: ReLU as the FFN activation.
 *
 * Conventions (all calls):
 *   - Matrices are row-major. bf16 = 16-bit brain float, passed as void*.
 *     Every pointer marked "device" is CUDA device memory on the current device.
 *   - The caller owns all memory. The library never allocates or frees device
 *     memory and never synchronises, except p24_query_status.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and returns a p24_status. Arguments are validated on the
 *     host before anything is launched; on an error nothing is launched.
 *   - Alignment: every device base pointer must be 16-byte aligned and every
 *     row stride must be a multiple of 16 bytes (P24_EALIGN otherwise).
 *   - 2:4 rule: in each group of 4 consecutive elements along the pruned axis,
 *     the two of largest magnitude are kept; magnitude is the bf16 bit pattern
 *     with the sign cleared, compared as an unsigned integer (so -0 == +0 and
 *     NaN sorts above inf); equal magnitudes go to the lower index.
 *   - The library is stateless apart from one device status word per GPU,
 *     written by kernels whose bounded waits expired (see p24_query_status).
 *   - The device addresses of the library's file-scope arrays (the status word,
 *     the scratch of p24_colsum_noalloc) are looked up once per device and kept
 *     for the life of the process. Resetting a device (cudaDeviceReset) after a
 *     call of this library ran on it is not supported: later calls would use
 *     the old context's addresses.
 */
#ifndef PRUNE24_H
#define PRUNE24_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  P24_OK = 0,
  P24_EINVAL = -1,        /* null pointer, bad shape, bad flag */
  P24_EALIGN = -2,        /* pointer or row stride not 16-byte aligned */
  P24_ECUDA = -3,         /* a CUDA runtime/driver call or launch failed */
  P24_ETIMEOUT = -4,      /* a kernel's bounded wait expired (device status word) */
  P24_EUNSUPPORTED = -5,  /* no sm_103a device, or a shape outside the supported set */
  P24_ENOSPACE = -6,      /* workspace smaller than required */
  P24_ECAPACITY = -7      /* a data-dependent output exceeded its capacity (device status word) */
} p24_status;

/*
 * A matrix pruned 2:4 along its columns, in compressed form (the "tailored
 * compressed storage format" of the ESPLAG success story, "Solution"; the
 * 2:4 case of values + 2-bit indices).
 *   rows, cols : logical dense shape; cols % 4 == 0.
 *   vals       : device bf16 [rows, ldv]. Group g of row r keeps two values,
 *                stored at vals[r*ldv + 2g] and [2g+1] in ascending index order.
 *                Entries from cols/2 to ldv-1 are zero padding.
 *   meta       : device uint8 [rows, ldm]. Group g's nibble i0 | (i1 << 2)
 *                (0 <= i0 < i1 <= 3 are the kept positions) sits in byte g/2,
 *                low nibble for even g. Unused nibbles up to ldm are 0x4.
 *   ldv        : >= p24_ld_vals(cols), multiple of 8 (16 bytes).
 *   ldm        : >= p24_ld_meta(cols), multiple of 16. The sparse GEMMs read
 *                16 metadata bytes per 128 columns, so this rounding is needed.
 */
typedef struct {
  void* vals;
  uint8_t* meta;
  int64_t rows;
  int64_t cols;
  int64_t ldv;
  int64_t ldm;
} p24_sparse;

/* Smallest legal strides of a compressed row of `cols` columns. */
int64_t p24_ld_vals(int64_t cols); /* round_up(cols/2, 8) elements */
int64_t p24_ld_meta(int64_t cols); /* 16 * ceil(cols/128) bytes */

/*
 * prune24_compress -- 2:4 magnitude pruning along the columns of W and
 * compression into values + metadata (ESPLAG success story, "Solution";
 * "To 2:4 Sparsity and Beyond", abstract: 2:4 for the weights).
 *   W       : device bf16 [rows, ldw], read only. cols % 4 == 0, ldw % 8 == 0.
 *   out     : descriptor of the output (vals/meta device buffers owned by the
 *             caller); out->rows == rows, out->cols == cols. All of vals and
 *             meta up to the strides is written, padding included.
 *   W_masked: optional device bf16 [rows, ldwm]: W with the pruned entries set
 *             to +0 (the dense form of the pruned matrix). NULL to skip.
 * Integer work only: the outputs are a pure function of the bits of W.
 */
int prune24_compress(const void* W, int64_t rows, int64_t cols, int64_t ldw,
                     const p24_sparse* out, void* W_masked, int64_t ldwm,
                     void* stream);

/*
 * prune24_transpose_repack -- the double prune of the SLOPE abstract: W_fwd
 * (given compressed, [N, K], 2:4 along K) is transposed to [K, N] and pruned
 * 2:4 again along N with the same rule, then compressed.
 *   fwd  : input descriptor, rows = N (N % 4 == 0), cols = K.
 *   bwdT : output descriptor, rows = K, cols = N. Written in full.
 * A column group with fewer than two nonzeros keeps zeros at the lowest free
 * indices, so the selected positions of bwdT need not lie inside the forward
 * mask, while its nonzero entries always do.
 */
int prune24_transpose_repack(const p24_sparse* fwd, const p24_sparse* bwdT,
                             void* stream);

/*
 * vnm24_compress -- V:2:M vector-wise N:M pruning (the VENOM format named in
 * the ESPLAG success story, "Solution"; v:n:m activation sparsity in the TO24
 * abstract). The pages give no layout, parameters or selection rule; this call
 * implements the following reading of them.
 *   - A [rows, cols] bf16 (row stride lda) is pruned along cols.
 *   - In every block of V consecutive rows (the last block may be shorter) and
 *     every group of M consecutive columns, the same 4 columns are kept for all
 *     rows of the block: the 4 with the largest L1 norm over the block (fp32
 *     sum, rows in order; compared as the sum's bit pattern, every NaN equal
 *     and above inf; ties to the lower column).
 *   - Each row then keeps 2 of its values at those 4 columns by the 2:4 rule of
 *     prune24_compress.
 *   V >= 1; M in {4, 8, 16, 32, 64, 128}; cols % M == 0. M = 4 is plain 2:4.
 * Outputs (caller-owned device memory):
 *   colidx : uint8 [ceil(rows/V), cols/M, 4], the kept column offsets (0..M-1)
 *            of each block and group, ascending.
 *   out    : descriptor of the condensed matrix, rows = rows, cols = 4*cols/M:
 *            row r, group g holds A's values at the 4 kept columns of g in the
 *            2:4 format of prune24_compress (values, nibbles, padding).
 *   A_masked : optional device bf16 [rows, ldam]: A with every pruned entry set
 *            to +0 (the dense form of the V:2:M matrix). It may be A itself
 *            (in place, ldam == lda). Needs V <= 256 and cols % 8 == 0
 *            (P24_EUNSUPPORTED otherwise). NULL to skip.
 * Returns P24_EINVAL for bad V, M, shapes or null pointers, P24_EALIGN for
 * misaligned A or out; nothing is launched then.
 */
int vnm24_compress(const void* A, int64_t rows, int64_t cols, int64_t lda,
                   int64_t V, int64_t M, uint8_t* colidx, const p24_sparse* out,
                   void* A_masked, int64_t ldam, void* stream);

/*
 * vnm24_spmm -- Y = act(A . B + bias) with A V:2:M-sparse, as vnm24_compress
 * writes it, and B dense with its reduction axis outermost (V:N:M activations
 * feeding the next FFN matmul: "To 2:4 Sparsity and Beyond", abstract; the
 * VENOM format of the ESPLAG success story, "Solution").
 *   colidx, A : vnm24_compress's outputs for an [R, K] matrix pruned with V and
 *            M (A->rows = R, A->cols = 4 K / M).
 *   B      : device bf16 [K, ldb], N columns, read only (for Y = A W^T, the
 *            weight W [N, K] stored transposed).
 *   bias   : device fp32 [N] with P24_EPI_BIAS; flags: P24_EPI_BIAS | P24_EPI_RELU.
 *   Y      : device bf16 [R, ldy], N columns; fp32 accumulation, one rounding.
 * Each block of V rows multiplies, per group of M, the 4 rows of B its colidx
 * selects (fetched by TMA gather), and the sparse tensor cores skip the 2 pruned
 * values of every 4: the result is the dense product of A's decompressed form and
 * B, up to the order of the fp32 sums.
 * Supported shapes (P24_EUNSUPPORTED otherwise): V a multiple of 256 (a CTA pair's
 * 256 rows share one selection), A->cols a multiple of 128 (K a multiple of 32 M),
 * N a multiple of 256. colidx must be 16-byte aligned (P24_EALIGN).
 */
int vnm24_spmm(const uint8_t* colidx, const p24_sparse* A, int64_t V, int64_t M,
               const void* B, int64_t N, int64_t ldb, const float* bias,
               uint32_t flags, void* Y, int64_t ldy, void* stream);

/*
 * prune24_compress_both -- prune24_compress followed by
 * prune24_transpose_repack in one pass over the dense W (the per-step mask
 * recompute of gradual magnitude pruning, ESPLAG success story, "Research
 * Topic"). rows % 4 == 0. Outputs are bit-identical to the two separate calls.
 */
int prune24_compress_both(const void* W, int64_t rows, int64_t cols, int64_t ldw,
                          const p24_sparse* fwd, const p24_sparse* bwdT,
                          void* W_masked, int64_t ldwm, void* stream);

/* Epilogue flags of the sparse GEMMs. */
#define P24_EPI_BIAS  0x1u  /* add an fp32 bias per output column */
#define P24_EPI_RELU  0x2u  /* ReLU after the bias (sets +0 for x <= 0) */
#define P24_EPI_ACT24 0x4u  /* 2:4-prune the bf16 output along its columns */
/* Test only (spmm24_fwd): the first CTA pair skips the loads of one pipeline stage,
 * so that the bounded waits of the real kernel expire; the call then leaves
 * P24_ETIMEOUT in the status word (see p24_query_timeout) and Y undefined. */
#define P24_EPI_TEST_STALL 0x80000000u

/*
 * spmm24_fwd -- forward linear with a 2:4 weight on the sparse tensor cores
 * (ESPLAG success story, "Research Topic": the SpMM):
 *   Y = act(X . W^T + bias), accumulated in fp32, rounded once to bf16.
 *   X     : device bf16 [M, ldx], K = W->cols columns.
 *   W     : compressed weight, rows = N (output features), cols = K.
 *   bias  : device fp32 [N] if flags has P24_EPI_BIAS, else ignored.
 *   flags : P24_EPI_BIAS | P24_EPI_RELU | P24_EPI_ACT24.
 *   Y     : device bf16 [M, ldy]. With P24_EPI_ACT24 it receives the pruned
 *           output (zeros off the activation mask).
 *   Y24   : with P24_EPI_ACT24, the compressed 2:4 form of Y along N
 *           ("To 2:4 Sparsity and Beyond": sparse activations); rows = M,
 *           cols = N (N % 4 == 0). NULL otherwise.
 * The 2:4 decision is taken on the rounded bf16 values.
 */
int spmm24_fwd(const void* X, int64_t M, int64_t ldx, const p24_sparse* W,
               const float* bias, uint32_t flags, void* Y, int64_t ldy,
               const p24_sparse* Y24, void* stream);

/*
 * spmm24_fwd_sparse_act -- forward linear whose INPUT is the 2:4-sparse
 * operand ("To 2:4 Sparsity and Beyond": sparse activations feeding the next
 * FFN matmul):
 *   Y = Xs . Wm^T + bias,   Xs compressed [M, K] (2:4 along K),
 *   Wm : device bf16 [N, ldw] dense weight (normally the weight on its own
 *        2:4 mask, as prune24_compress's W_masked writes it).
 *   flags : P24_EPI_BIAS | P24_EPI_RELU.
 */
int spmm24_fwd_sparse_act(const p24_sparse* Xs, const void* Wm, int64_t N,
                          int64_t ldw, const float* bias, uint32_t flags,
                          void* Y, int64_t ldy, void* stream);

/*
 * spmm24_bwd_dx -- input gradient through a double-pruned weight (SLOPE
 * abstract):  dX = (dY . W_bwd) * [gate > 0].
 *   dY    : device bf16 [M, lddy], N = WbwdT->cols columns.
 *   WbwdT : compressed W_bwd^T, rows = K, cols = N (2:4 along N), as
 *           prune24_transpose_repack writes it.
 *   gate  : optional device bf16 [M, ldg] (the forward ReLU output); where
 *           gate <= 0 the gradient is 0 (ReLU'(0) = 0). NULL = no gate.
 *   dX    : device bf16 [M, lddx], K columns.
 *   dbias : optional device fp32 [K], 16-byte aligned: receives the bias
 *           gradient of the layer below, dbias[k] = sum over m of dX[m, k]
 *           (the stored bf16 values), fused into the GEMM's epilogue. It is
 *           zeroed on `stream` and then accumulated with fp32 atomics, so the
 *           summation order (and the last bits) may differ from run to run;
 *           p24_colsum gives a fixed-order sum. NULL = not computed.
 */
int spmm24_bwd_dx(const void* dY, int64_t M, int64_t lddy, const p24_sparse* WbwdT,
                  const void* gate, int64_t ldg, void* dX, int64_t lddx,
                  float* dbias, void* stream);

/*
 * Low-rank adapters (SLOPE abstract: "low-rank adapters" added beside the
 * double-pruned sparse weights for the final iterations of pretraining). Read
 * as a dense rank-r term per linear: Y = X W_s^T + (X R^T) L^T with L [N, r],
 * R [r, K], trained with its exact gradients. The two products of rank r are
 * computed once per call with p24_gemm_nt; the sparse GEMMs then add them as
 * r / 64 extra dense K-steps into the same fp32 accumulator, before the epilogue.
 * r > 0 and r % 8 == 0 (16-byte rows). Memory is the caller's, as everywhere.
 *
 * spmm24_fwd_lowrank -- spmm24_fwd plus the adapter:
 *   Y = act(X W^T + T L^T + bias),  T : device bf16 [M, ldt] = X R^T (r columns),
 *   L : device bf16 [N, ldl] (r columns), N = W->rows.  Other arguments as spmm24_fwd.
 */
int spmm24_fwd_lowrank(const void* X, int64_t M, int64_t ldx, const p24_sparse* W,
                       const void* T, int64_t ldt, const void* L, int64_t ldl, int64_t r,
                       const float* bias, uint32_t flags, void* Y, int64_t ldy,
                       const p24_sparse* Y24, void* stream);

/*
 * spmm24_bwd_dx_lowrank -- spmm24_bwd_dx plus the adapter's input gradient:
 *   dX = (dY W_bwd + U R) * [gate > 0],  U : device bf16 [M, ldu] = dY L
 *   (r columns), Rt : device bf16 [K, ldrt] = R^T (r columns), K = WbwdT->rows.
 *   Other arguments (gate, dbias) as spmm24_bwd_dx.
 */
int spmm24_bwd_dx_lowrank(const void* dY, int64_t M, int64_t lddy, const p24_sparse* WbwdT,
                          const void* U, int64_t ldu, const void* Rt, int64_t ldrt, int64_t r,
                          const void* gate, int64_t ldg, void* dX, int64_t lddx,
                          float* dbias, void* stream);

/*
 * p24_gemm_nt -- C = A B^T, the adapters' rank-r products (T = X R^T, U = dY L
 * with L^T as B): A device bf16 [M, lda], B [N, ldb], both K columns; C bf16
 * [M, ldc]; fp32 accumulation, one rounding. Runs on the sparse GEMM's pipeline
 * with dense stages only.
 */
int p24_gemm_nt(const void* A, int64_t M, int64_t lda, const void* B, int64_t N,
                int64_t ldb, int64_t K, void* C, int64_t ldc, void* stream);

/*
 * p24_gemm_tn -- C = A^T B, a contraction over the M tokens, unmasked: the
 * adapters' weight gradients (dL = dY^T T, dR = U^T X). A device bf16 [M, lda]
 * (N columns), B [M, ldb] (K columns), C bf16 [N, ldc] (K columns). Runs on the
 * weight-gradient kernel with the mask off.
 */
int p24_gemm_tn(const void* A, int64_t lda, const void* B, int64_t ldb, int64_t M,
                int64_t N, int64_t K, void* C, int64_t ldc, void* stream);

/* p24_transpose -- dst [cols, ldd] = src [rows, lds]^T, bf16 (L^T and R^T for the
 * adapters' backward products). Any strides (lds >= cols, ldd >= rows); 2-byte
 * aligned pointers. */
int p24_transpose(const void* src, int64_t rows, int64_t cols, int64_t lds, void* dst,
                  int64_t ldd, void* stream);

/*
 * masked_dw_gemm -- weight gradient of a 2:4 linear, kept on the forward mask:
 *   dW = (dY^T . X) * mask(Wfwd), a dense contraction over M in fp32.
 *   dY   : device bf16 [M, lddy], N columns;  X : device bf16 [M, ldx], K columns.
 *   Wfwd : the forward weight's descriptor; only its meta is read (N rows, K cols).
 *   dW   : device bf16 [N, lddw]; entries off the mask are written as +0.
 */
int masked_dw_gemm(const void* dY, int64_t lddy, const void* X, int64_t ldx,
                   int64_t M, const p24_sparse* Wfwd, void* dW, int64_t lddw,
                   void* stream);

/*
 * p24_colsum -- bias gradient: out[n] = sum over m of G[m, n] (fp32 result,
 * fp32 partial sums combined in a fixed order, so repeated calls are
 * bit-identical).
 *   G   : device bf16 [M, ldg], N columns;  out : device fp32 [N].
 *   ws  : device scratch of at least p24_colsum_workspace_size(M, N) bytes.
 */
size_t p24_colsum_workspace_size(int64_t M, int64_t N);
int p24_colsum(const void* G, int64_t M, int64_t N, int64_t ldg, float* out,
               void* ws, size_t ws_bytes, void* stream);

/*
 * p24_colsum_noalloc -- p24_colsum for callers that cannot allocate device
 * memory. The pages have no counterpart to this call; it exists for integration.
 *
 * Who needs it: a caller that has no device allocator of its own to call, e.g.
 * C code embedded in a framework whose memory pool already owns the GPU's memory
 * (a cudaMalloc behind the pool's back fails or fragments it), or code on a path
 * where a cudaMalloc/cudaFree, which can synchronise the device, would stall the
 * asynchronous pipeline around it.
 *
 * How: the partial sums go to a fixed array of P24_COLSUM_NOALLOC_SCRATCH_FLOATS
 * floats (4 MiB) inside the library, held on every GPU that loads the library
 * until the process exits. The call allocates and frees nothing.
 *   G, M, N, ldg, out : as p24_colsum. Results equal p24_colsum's up to fp32
 *                       rounding (for very wide N fewer row slabs are used);
 *                       repeated calls with the same input are bit-identical.
 *   N > P24_COLSUM_NOALLOC_MAX_COLS is rejected with P24_ENOSPACE (nothing launched).
 * The first call on each device looks up the scratch array's device address
 * (with that device current); make that first call before any stream capture.
 * Every call uses the same scratch array and leaves its partial sums there;
 * calls whose kernels overlap on the GPU (different streams, no ordering) race
 * on it and give wrong sums: order them on one stream or with events.
 */
#define P24_COLSUM_NOALLOC_SCRATCH_FLOATS (1 << 20)
#define P24_COLSUM_NOALLOC_MAX_COLS P24_COLSUM_NOALLOC_SCRATCH_FLOATS
int p24_colsum_noalloc(const void* G, int64_t M, int64_t N, int64_t ldg, float* out, void* stream);

/*
 * Hybrid ELL + dense-overflow activations ("Sparser, Faster, Lighter Transformer
 * Language Models", "Methodologie": for training, rows with few nonzeros are held in
 * a compact ELL matrix and rows with many -- overflows -- in a dense backup matrix;
 * custom kernels multiply hybrid by dense and dense into hybrid). The page gives no
 * layout; this is the one used here. A [rows, cols] bf16, a value is nonzero when its
 * magnitude bits are not 0 (-0 is zero):
 *   nnz      : device int32 [rows], the nonzero count of each row.
 *   ell_cols : device uint16 [rows, E]; ell_vals : device bf16 [rows, E]. A row with
 *              nnz <= E keeps its nonzero columns in ascending order and their values;
 *              the other slots (and every slot of an overflow row) hold column 0, +0.
 *   slot     : device int32 [rows]: -1 for an ELL row, else the row's rank among the
 *              overflow rows (nnz > E), in row order.
 *   ovf_rows : device int32 [cap], the overflow rows by slot (-1 past their count).
 *   n_ovf    : device int32 [1], the number of overflow rows (it may exceed cap).
 *   ovf      : device bf16 [cap, ldo]: backup row k = overflow row ovf_rows[k] as it is.
 * E >= 1; cols <= 65536 and cols % 8 == 0; cap >= 0. 16-byte aligned pointers, except
 * nnz, slot, ovf_rows, n_ovf (4-byte). More overflow rows than cap is an error found on
 * the device: the rows past the capacity are not stored, the products write zeros for
 * them, and P24_ECAPACITY is left in the status word (p24_query_status).
 */
typedef struct {
  int64_t rows, cols, E, cap;
  int32_t* nnz;
  uint16_t* ell_cols;
  void* ell_vals;
  int32_t* slot;
  int32_t* ovf_rows;
  int32_t* n_ovf;
  void* ovf;
  int64_t ldo;
} p24_hybrid;

/* hyb_compress -- the hybrid form of A (device bf16 [h->rows, lda], h->cols columns),
 * written into h's buffers (caller-owned). Integer work: a pure function of A's bits. */
int hyb_compress(const void* A, int64_t lda, const p24_hybrid* h, void* stream);

/* hyb_spmm -- hybrid to dense: Y = A . B, A in hybrid form [rows, cols], B device bf16
 * [cols, ldb] with N columns (e.g. W_down^T for the down projection, W_up for the input
 * gradient), Y device bf16 [rows, ldy]; fp32 accumulation, one rounding. N % 8 == 0. */
int hyb_spmm(const p24_hybrid* h, const void* B, int64_t N, int64_t ldb, void* Y, int64_t ldy, void* stream);

/* hyb_sddmm -- dense to hybrid: S = (G . B^T) at A's nonzero positions, in A's hybrid
 * layout (dH = (dY W_down) * [H != 0] with G = dY, B = W_down^T). G device bf16
 * [rows, ldg], B device bf16 [cols, ldb], both N columns (N % 8 == 0). Outputs:
 * S_ell bf16 [rows, E] (values in A's ELL slots, +0 padding) and S_ovf bf16 [cap, lds]
 * (backup rows: values at A's nonzeros, +0 elsewhere). fp32 accumulation. */
int hyb_sddmm(const p24_hybrid* h, const void* G, int64_t N, int64_t ldg, const void* B, int64_t ldb,
              void* S_ell, void* S_ovf, int64_t lds, void* stream);

/* Flags of ffn24_step. */
#define P24_STEP_ACT24 0x1u /* 2:4-prune ReLU(up) and feed it as the sparse operand of down */
#define P24_STEP_KEEP_MASKS 0x2u /* use the caller's compressed weights as they are (fixed masks) */
#define P24_STEP_ADAPTERS 0x4u /* SLOPE's low-rank adapters on both linears (rank r) */
#define P24_STEP_VNM 0x8u /* V:2:M-prune ReLU(up) along ffn and feed it to the down GEMM (vnm24_spmm) */

/*
 * One FFN layer (up -> ReLU -> down), forward and backward, every matmul 2:4
 * ("To 2:4 Sparsity and Beyond", abstract; ESPLAG "Research Topic"; SLOPE):
 *   prune W_up, W_down 2:4 along their reduction axis and double-prune their
 *   transposes (fresh masks every step);
 *   H  = ReLU(X W_up^T + b_up)           (ACT24: H pruned 2:4 along ffn)
 *   Y  = H W_down^T + b_down
 *   dH = (dY W_down_bwd) * [H > 0];  db_up = colsum(dH);  db_down = colsum(dY)
 *   (db_up is fused into the dH epilogue with fp32 atomics, so its last bits may
 *   vary from run to run; db_down is a fixed-order sum)
 *   dW_down = (dY^T H) on mask(W_down);  dX = dH W_up_bwd;  dW_up = (dH^T X) on mask(W_up)
 * All tensors are dense, row-major, contiguous (row stride = column count):
 *   X, dY, Y, dX : bf16 [M, d];  W_up, dW_up : bf16 [ffn, d];
 *   W_down, dW_down : bf16 [d, ffn];  H : bf16 [M, ffn] (output, the stored
 *   activation); b_up, db_up : fp32 [ffn];  b_down, db_down : fp32 [d].
 *   b_up / b_down may be NULL (no bias); db_up / db_down may be NULL.
 * d % 8 == 0 and ffn % 8 == 0.
 * Compressed weights (caller buffers, optional unless P24_STEP_KEEP_MASKS):
 *   up_fwd [ffn, d] and down_fwd [d, ffn]: the forward 2:4 weights;
 *   up_bwdT [d, ffn] and down_bwdT [ffn, d]: their double-pruned transposes;
 *   W_down_masked : bf16 [d, ffn] (row stride ffn), W_down on its 2:4 mask, the
 *   dense operand of the down GEMM under P24_STEP_ACT24.
 *   Without P24_STEP_KEEP_MASKS (gradual magnitude pruning, ESPLAG "Research
 *   Topic"): the step prunes W_up and W_down afresh and writes the results to
 *   these buffers where given (NULL: kept in the workspace).
 *   With P24_STEP_KEEP_MASKS (fixed masks): the step reads them as they are,
 *   prunes nothing and does not read W_up / W_down (which may be NULL); the four
 *   compressed buffers (and W_down_masked under P24_STEP_ACT24) are required.
 * Low-rank adapters (P24_STEP_ADAPTERS; see spmm24_fwd_lowrank): each linear
 *   gains a dense rank-r term, the up one X R_up^T L_up^T and the down one
 *   H R_down^T L_down^T, trained with exact gradients:
 *   L_up [ffn, r], R_up [r, d], L_down [d, r], R_down [r, ffn] (bf16, contiguous)
 *   and their gradients dL_up, dR_up, dL_down, dR_down of the same shapes:
 *     T_up = X R_up^T;  H = ReLU(X W_up^T + T_up L_up^T + b_up);
 *     T_dn = H R_down^T;  Y = H W_down^T + T_dn L_down^T + b_down;
 *     U_dn = dY L_down;  dH = (dY W_down_bwd + U_dn R_down) * [H > 0];
 *     U_up = dH L_up;  dX = dH W_up_bwd + U_up R_up;
 *     dL_down = dY^T T_dn;  dR_down = U_dn^T H;  dL_up = dH^T T_up;  dR_up = U_up^T X
 *   (T and U rounded to bf16). r > 0, r % 8 == 0; the workspace size then comes
 *   from ffn24_workspace_size_lowrank.
 * dH (optional): device bf16 [M, ffn] (row stride ffn). Where given, the step
 *   stores the gated hidden gradient dH (the bf16 operand of dX and dW_up) there
 *   instead of in the workspace, so the caller can read it afterwards. NULL: the
 *   workspace holds it.
 * V:N:M activations (P24_STEP_VNM; "To 2:4 Sparsity and Beyond", abstract: v:n:m
 *   sparsity for the activations): H is pruned V:2:M along ffn by vnm24_compress's
 *   rule with V = vnm_V and M = vnm_M, in place (the H output is the pruned H), and
 *   the down forward runs on the sparse tensor cores as vnm24_spmm with W_down on
 *   its 2:4 mask, transposed, as the gathered operand:
 *     H = V:2:M(ReLU(X W_up^T + b_up));  Y = H W_down^T + b_down;
 *   the backward is the one above with this H (the gate [H > 0] is the V:2:M mask
 *   times the ReLU gate). Requires vnm_V = 256, vnm_M in {4, 8, ..., 128},
 *   ffn % (32 vnm_M) == 0 and d % 256 == 0; not with P24_STEP_ACT24 or
 *   P24_STEP_ADAPTERS (P24_EUNSUPPORTED). The workspace size comes from
 *   ffn24_workspace_size_args.
 */
typedef struct {
  int64_t M, d, ffn;
  uint32_t flags;
  const void* X;
  const void* W_up;
  const float* b_up;
  const void* W_down;
  const float* b_down;
  const void* dY;
  void* Y;
  void* H;
  void* dX;
  void* dW_up;
  void* dW_down;
  float* db_up;
  float* db_down;
  p24_sparse* up_fwd;
  p24_sparse* up_bwdT;
  p24_sparse* down_fwd;
  p24_sparse* down_bwdT;
  void* W_down_masked;
  int64_t r;
  const void* L_up;
  const void* R_up;
  const void* L_down;
  const void* R_down;
  void* dL_up;
  void* dR_up;
  void* dL_down;
  void* dR_down;
  void* dH;
  int64_t vnm_V;
  int64_t vnm_M;
} p24_ffn_args;

/* Device workspace ffn24_step needs for these sizes (compressed weights, dH, ...). */
size_t ffn24_workspace_size(int64_t M, int64_t d, int64_t ffn, uint32_t flags);
/* The same for the step described by a (M, d, ffn, flags, r, vnm_V, vnm_M are read):
 * covers every flag, P24_STEP_VNM included. 0 for invalid sizes. */
size_t ffn24_workspace_size_args(const p24_ffn_args* a);
/* The same with low-rank adapters of rank r (flags with P24_STEP_ADAPTERS). */
size_t ffn24_workspace_size_lowrank(int64_t M, int64_t d, int64_t ffn, uint32_t flags, int64_t r);
int ffn24_step(const p24_ffn_args* a, void* workspace, size_t ws_bytes, void* stream);

/*
 * ffn24_step_traced -- ffn24_step that also records caller-created CUDA events
 * (cudaEvent_t handles) on `stream` around each phase of the step, for
 * per-kernel timing without a synchronisation: events[2p] before and
 * events[2p+1] after phase p, for p < min(P24_STEP_PHASES, n_events / 2).
 * Phases: 0 prune+double-prune W_up, 1 the same for W_down (both empty with
 * P24_STEP_KEEP_MASKS), 2 up forward (H),
 * 3 down forward (Y), 4 down backward dX (dH and db_up), 5 db_down, 6 dW_down,
 * 7 up backward dX, 8 dW_up. events may be NULL (then identical to ffn24_step).
 */
#define P24_STEP_PHASES 9
int ffn24_step_traced(const p24_ffn_args* a, void* workspace, size_t ws_bytes, void* stream,
                      void* const* events, int n_events);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t p24_launch_count(void);

/*
 * p24_query_status -- synchronise `stream`, then return and clear the device
 * status word of the current GPU: P24_OK, or P24_ETIMEOUT if a kernel gave up
 * a bounded wait (the kernel then skipped its remaining work and exited
 * cleanly, so the context stays usable).
 */
int p24_query_status(void* stream);

/*
 * p24_selftest_timeout -- exercise the failure path of the bounded waits: one
 * kernel waits up to limit_ns (0 < limit_ns <= 1e10) on a barrier that nothing
 * arrives on, records P24_ETIMEOUT in the device status word and returns
 * normally. A following p24_query_status(stream) returns P24_ETIMEOUT (and
 * clears it); the context stays usable. Nothing is faulted, trapped or hung.
 */
int p24_selftest_timeout(int64_t limit_ns, void* stream);

/*
 * p24_query_timeout -- p24_query_status that also reports where the first
 * expired wait happened: *cta = its CTA (blockIdx.x) and *barrier = the shared
 * memory address of the mbarrier it waited on, as that CTA saw it (the offset in
 * the low 24 bits; a CTA of a cluster has its rank above them). Both are -1 when
 * the status is P24_OK. Either pointer may be NULL. Clears the status.
 */
int p24_query_timeout(void* stream, int64_t* cta, int64_t* barrier);

/* Static text for a p24_status code. */
const char* p24_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* PRUNE24_H */
