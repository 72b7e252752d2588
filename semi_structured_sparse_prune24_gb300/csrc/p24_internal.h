// p24_internal.h -- host-side launchers shared between the translation units
// of libprune24 (not part of the public ABI; see include/prune24.h).
#pragma once
#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "prune24.h"

namespace p24 {

// ---- pruning / packing (prune24_kernels.cu) ----
cudaError_t launch_compress(const void* W, int64_t rows, int64_t cols, int64_t ldw, const p24_sparse& out,
                            void* W_masked, int64_t ldwm, cudaStream_t s);
// W_masked_T (optional, not together with W_masked): the forward-masked W transposed, [cols, ldwmT].
cudaError_t launch_compress_both(const void* W, int64_t rows, int64_t cols, int64_t ldw, const p24_sparse& fwd,
                                 const p24_sparse& bwdT, void* W_masked, int64_t ldwm, cudaStream_t s,
                                 void* W_masked_T = nullptr, int64_t ldwmT = 0);
// W_masked_T (optional): the forward-masked matrix transposed, [fwd.cols, ldwmT].
cudaError_t launch_transpose_repack(const p24_sparse& fwd, const p24_sparse& bwdT, cudaStream_t s,
                                    void* W_masked_T = nullptr, int64_t ldwmT = 0);
cudaError_t launch_pad(const p24_sparse& d, cudaStream_t s);
int64_t colsum_slabs(int64_t M);
cudaError_t launch_selftest_timeout(uint64_t limit_ns, int* status, cudaStream_t s);
cudaError_t launch_colsum(const void* G, int64_t M, int64_t N, int64_t ldg, float* out, float* ws, cudaStream_t s);
// The step's db_down: more row slabs for short inputs; scratch of colsum_step_slabs(M, N) * N floats.
int64_t colsum_step_slabs(int64_t M, int64_t N);
cudaError_t launch_colsum_step(const void* G, int64_t M, int64_t N, int64_t ldg, float* out, float* ws,
                               cudaStream_t s);
// Same sums with the library's fixed device scratch instead of a caller workspace.
constexpr int64_t kNoAllocColsumScratch = P24_COLSUM_NOALLOC_SCRATCH_FLOATS;  // floats (4 MiB per GPU)
static_assert(P24_COLSUM_NOALLOC_MAX_COLS <= P24_COLSUM_NOALLOC_SCRATCH_FLOATS,
              "the widest accepted input needs one row slab of partial sums");
cudaError_t launch_colsum_noalloc(const void* G, int64_t M, int64_t N, int64_t ldg, float* out, cudaStream_t s);

// ---- tensor-core GEMMs (gemm24_kernels.cu) ----
struct EpiArgs {
  const float* bias = nullptr;  // fp32 per output column (of Y), or null
  bool relu = false;
  const void* gate = nullptr;   // bf16 [M, ldg] ReLU output for the backward gate, or null
  int64_t ldg = 0;
  float* dbias = nullptr;              // += column sums of the stored output (transposed output only)
  // low-rank term added to the product before the epilogue: lr_a [rows of A, r] . lr_b [rows of B, r]^T
  const void* lr_a = nullptr;
  int64_t lr_lda = 0;
  const void* lr_b = nullptr;
  int64_t lr_ldb = 0;
  int64_t lr_r = 0;
  bool test_stall = false;  // test only: the first CTA pair skips one stage's loads (its waits expire)
  p24_sparse act24{};           // compressed activation output (vals != null => enabled)
};

// C[i, j] = sum_r A[i, r] * B[j, r] with A 2:4-sparse (compressed, K-major) and
// B dense K-major; written transposed (out[j, i]) when `transposed_out`.
cudaError_t launch_spmm(const p24_sparse& A, const void* B, int64_t rowsB, int64_t ldb, void* out,
                        int64_t ldo, bool transposed_out, const EpiArgs& epi, int* status, cudaStream_t s);

// Y [R, N] = act(A . B + bias) with A V:2:M-sparse (colidx [ceil(R/V), K/Mg, 4] and the
// condensed 2:4 descriptor, cols = 4 K / Mg) and B dense K-outer [K, ldb]. Requires
// V % 256 == 0, A.cols % 128 == 0 and N % 256 == 0 (checked by the caller).
cudaError_t launch_vnm_compress(const void* A, int64_t rows, int64_t cols, int64_t lda, int V, int M,
                                uint8_t* colidx, const p24_sparse& out, void* A_masked, int64_t ldam, cudaStream_t s);
cudaError_t launch_vnm_spmm(const uint8_t* colidx, const p24_sparse& A, int V, int Mg, const void* B, int64_t N,
                            int64_t ldb, const float* bias, bool relu, void* Y, int64_t ldy, int* status,
                            cudaStream_t s);

// dW[n, k] = sum_m dY[m, n] * X[m, k] on mask(meta) (both operands MN-major).
// C [M, N] = A [M, K] . B [N, K]^T, bf16 in and out, fp32 accumulation (K-major operands).
cudaError_t launch_gemm_nt(const void* A, int64_t M, int64_t lda, const void* B, int64_t N, int64_t ldb, int64_t K,
                           void* C, int64_t ldc, int* status, cudaStream_t s);
// C [N, K] = A [M, N]^T . B [M, K] (contraction over M), bf16 out, no mask.
cudaError_t launch_gemm_tn(const void* A, int64_t lda, const void* B, int64_t ldb, int64_t M, int64_t N, int64_t K,
                           void* C, int64_t ldc, int* status, cudaStream_t s);
// dst [cols, rows] = src [rows, cols]^T, bf16.
cudaError_t launch_transpose_bf16(const void* src, int64_t rows, int64_t cols, int64_t lds, void* dst, int64_t ldd,
                                  cudaStream_t s);
// Extra output of a masked dW launch, computed unmasked from the same pass: a second
// A operand a2 [M, n2] gives out2 [n2, K] = a2^T . X (it shares X's panels), or a second
// B operand b2 [M, k2] gives out2 [N, k2] = dY^T . b2 (it shares dY's panels).
struct DwExtra {
  const void* a2 = nullptr;
  int64_t lda2 = 0, n2 = 0;
  const void* b2 = nullptr;
  int64_t ldb2 = 0, k2 = 0;
  void* out2 = nullptr;
  int64_t ldo2 = 0;
};
cudaError_t launch_masked_dw_extra(const void* dY, int64_t lddy, const void* X, int64_t ldx, int64_t M, int64_t N,
                                   int64_t K, const uint8_t* meta, int64_t ldm, void* dW, int64_t lddw,
                                   const DwExtra& ex, int* status, cudaStream_t s);
cudaError_t launch_masked_dw(const void* dY, int64_t lddy, const void* X, int64_t ldx, int64_t M, int64_t N,
                             int64_t K, const uint8_t* meta, int64_t ldm, void* dW, int64_t lddw, int* status,
                             cudaStream_t s);

// ---- hybrid ELL + dense-overflow activations (hyb_kernels.cu)
cudaError_t launch_hyb_compress(const void* A, int64_t lda, const p24_hybrid& h, int* status, cudaStream_t s);
cudaError_t launch_hyb_spmm(const p24_hybrid& h, const void* B, int64_t N, int64_t ldb, void* Y, int64_t ldy,
                            cudaStream_t s);
cudaError_t launch_hyb_sddmm(const p24_hybrid& h, const void* G, int64_t N, int64_t ldg, const void* B, int64_t ldb,
                             void* S_ell, void* S_ovf, int64_t lds, cudaStream_t s);

// A 2-D tensor map over a row-major matrix, for the HBM-bound kernels' TMA staging:
// `inner` columns of `outer` rows, boxes of box_inner x box_outer; swizzle128 lays each
// 128-byte box row out with the 128B swizzle (box_inner x element size must be 128).
bool make_tensor_map_2d(CUtensorMap* m, bool bf16, const void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128 = false);

int* device_status_ptr();  // the status word of the current device

// Launch with programmatic stream serialization: the kernel may start while the
// stream's previous kernel finishes, and must call pdl_wait() before touching global
// memory (p24_ptx.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
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
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// The same launch without the attribute (stream order as usual). Measured: the fused
// prune + double prune is faster launched this way (the 70B tail step 2.03 -> 1.97 ms
// against programmatic launch), while the GEMMs and column sums gain from it.
template <typename... KArgs, typename... Args>
cudaError_t launch_plain(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                         Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Count one kernel launch (called by every launcher after a successful launch).
void count_launch();

}  // namespace p24
