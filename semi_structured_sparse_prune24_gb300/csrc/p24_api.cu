// p24_api.cu -- the extern "C" entry points of libprune24 declared in
// include/prune24.h: host-side validation (nothing is launched on an error),
// workspace carving for the FFN step, and the device status word.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <cstdint>
#include <cstring>

#include "p24_internal.h"

namespace p24 {
namespace {

// [0] P24_OK, or P24_ETIMEOUT after a bounded wait expired; [1] the CTA and [2] the
// barrier's shared address of the first expired wait; [3] unused
__device__ int g_status[4];

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dense(const void* p, int64_t rows, int64_t cols, int64_t ld) {
  if (rows < 0 || cols < 0 || rows > kMaxDim || cols > kMaxDim) return P24_EINVAL;
  if (rows == 0 || cols == 0) return P24_OK;
  if (!p) return P24_EINVAL;
  if (ld < cols) return P24_EINVAL;
  if (!aligned16(p) || (ld % 8) != 0) return P24_EALIGN;
  return P24_OK;
}

int check_sparse(const p24_sparse* d) {
  if (!d) return P24_EINVAL;
  if (d->rows < 0 || d->cols < 0 || d->rows > kMaxDim || d->cols > kMaxDim) return P24_EINVAL;
  if (d->cols % 4 != 0) return P24_EINVAL;
  if (d->rows == 0 || d->cols == 0) return P24_OK;
  if (!d->vals || !d->meta) return P24_EINVAL;
  if (d->ldv < p24_ld_vals(d->cols) || d->ldm < p24_ld_meta(d->cols)) return P24_EINVAL;
  if (!aligned16(d->vals) || !aligned16(d->meta) || d->ldv % 8 != 0 || d->ldm % 16 != 0) return P24_EALIGN;
  return P24_OK;
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? P24_OK : P24_ECUDA; }

#define P24_TRY(expr)              \
  do {                             \
    const int _rc = (expr);        \
    if (_rc != P24_OK) return _rc; \
  } while (0)

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace of ffn24_step, carved in this order (each region 256-byte aligned).
struct StepLayout {
  p24_sparse up_fwd, up_bwdT, dn_fwd, dn_bwdT, hs;
  uint8_t* colidx;  // V:N:M: H's kept column offsets [ceil(M/V), ffn/vM, 4]
  void* wdmT;       // V:N:M: W_down on its 2:4 mask, transposed [ffn, d]
  // low-rank adapters: T_up, T_dn, U_dn, U_up [M, r]; Lt_up [r, ffn], Lt_dn [r, d], Rt_up [d, r], Rt_dn [ffn, r]
  void *T_up, *T_dn, *U_dn, *U_up, *Lt_up, *Lt_dn, *Rt_up, *Rt_dn;
  size_t off[16];
  size_t total;
};

void step_layout(int64_t M, int64_t d, int64_t ffn, uint32_t flags, int64_t r, char* base, StepLayout& L,
                 void** wdm, void** dH, float** cs, int64_t vV = 0, int64_t vM = 0) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + off : nullptr;
    off = round_up(off + bytes, 256);
    return static_cast<void*>(p);
  };
  auto sparse = [&](p24_sparse& s, int64_t rows, int64_t cols) {
    s.rows = rows;
    s.cols = cols;
    s.ldv = p24_ld_vals(cols);
    s.ldm = p24_ld_meta(cols);
    s.vals = take(static_cast<size_t>(rows * s.ldv * 2));
    s.meta = static_cast<uint8_t*>(take(static_cast<size_t>(rows * s.ldm)));
  };
  sparse(L.up_fwd, ffn, d);
  sparse(L.up_bwdT, d, ffn);
  sparse(L.dn_fwd, d, ffn);
  sparse(L.dn_bwdT, ffn, d);
  L.colidx = nullptr;
  L.wdmT = nullptr;
  if (flags & P24_STEP_ACT24) {
    sparse(L.hs, M, ffn);
    *wdm = take(static_cast<size_t>(d * ffn * 2));
  } else if ((flags & P24_STEP_VNM) && vV > 0 && vM > 0) {
    sparse(L.hs, M, 4 * (ffn / vM));  // the condensed H
    L.colidx = static_cast<uint8_t*>(take(static_cast<size_t>((M + vV - 1) / vV * (ffn / vM) * 4)));
    L.wdmT = take(static_cast<size_t>(d * ffn * 2));
    *wdm = nullptr;
  } else {
    std::memset(&L.hs, 0, sizeof(L.hs));
    *wdm = nullptr;
  }
  *dH = take(static_cast<size_t>(M * ffn * 2));
  if ((flags & P24_STEP_ADAPTERS) && r > 0) {
    const size_t mr = static_cast<size_t>(M * r * 2);
    L.T_up = take(mr);
    L.T_dn = take(mr);
    L.U_dn = take(mr);
    L.U_up = take(mr);
    L.Lt_up = take(static_cast<size_t>(r * ffn * 2));
    L.Lt_dn = take(static_cast<size_t>(r * d * 2));
    L.Rt_up = take(static_cast<size_t>(d * r * 2));
    L.Rt_dn = take(static_cast<size_t>(ffn * r * 2));
  } else {
    L.T_up = L.T_dn = L.U_dn = L.U_up = L.Lt_up = L.Lt_dn = L.Rt_up = L.Rt_dn = nullptr;
  }
  // db_down's partial sums (colsum_step_slabs(M, d) row slabs of d floats)
  *cs = static_cast<float*>(take(static_cast<size_t>(colsum_step_slabs(M, d) * d * 4)));
  L.total = off;
}

}  // namespace

std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int* device_status_ptr() {
  // the status word's device address, looked up once per device
  constexpr int kDevs = 64;
  static std::once_flag once[kDevs];
  static int* addr[kDevs] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return nullptr;
  std::call_once(once[dev], [dev] {
    int* p = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_status) == cudaSuccess) addr[dev] = p;
  });
  return addr[dev];
}

}  // namespace p24

using namespace p24;

extern "C" {

int64_t p24_ld_vals(int64_t cols) { return ((cols / 2) + 7) / 8 * 8; }
int64_t p24_ld_meta(int64_t cols) { return 16 * ((cols + 127) / 128); }

int prune24_compress(const void* W, int64_t rows, int64_t cols, int64_t ldw, const p24_sparse* out, void* W_masked,
                     int64_t ldwm, void* stream) {
  if (cols % 4 != 0) return P24_EINVAL;
  P24_TRY(check_dense(W, rows, cols, ldw));
  P24_TRY(check_sparse(out));
  if (out->rows != rows || out->cols != cols) return P24_EINVAL;
  if (W_masked) P24_TRY(check_dense(W_masked, rows, cols, ldwm));
  return cuda_status(launch_compress(W, rows, cols, ldw, *out, W_masked, ldwm, as_stream(stream)));
}

int prune24_transpose_repack(const p24_sparse* fwd, const p24_sparse* bwdT, void* stream) {
  P24_TRY(check_sparse(fwd));
  P24_TRY(check_sparse(bwdT));
  if (fwd->rows % 4 != 0) return P24_EINVAL;
  if (bwdT->rows != fwd->cols || bwdT->cols != fwd->rows) return P24_EINVAL;
  return cuda_status(launch_transpose_repack(*fwd, *bwdT, as_stream(stream)));
}

int prune24_compress_both(const void* W, int64_t rows, int64_t cols, int64_t ldw, const p24_sparse* fwd,
                          const p24_sparse* bwdT, void* W_masked, int64_t ldwm, void* stream) {
  if (cols % 4 != 0 || rows % 4 != 0) return P24_EINVAL;
  P24_TRY(check_dense(W, rows, cols, ldw));
  P24_TRY(check_sparse(fwd));
  P24_TRY(check_sparse(bwdT));
  if (fwd->rows != rows || fwd->cols != cols || bwdT->rows != cols || bwdT->cols != rows) return P24_EINVAL;
  if (W_masked) P24_TRY(check_dense(W_masked, rows, cols, ldwm));
  return cuda_status(launch_compress_both(W, rows, cols, ldw, *fwd, *bwdT, W_masked, ldwm, as_stream(stream)));
}

int vnm24_compress(const void* A, int64_t rows, int64_t cols, int64_t lda, int64_t V, int64_t M, uint8_t* colidx,
                   const p24_sparse* out, void* A_masked, int64_t ldam, void* stream) {
  if (V < 1 || V > kMaxDim) return P24_EINVAL;
  if (M < 4 || M > 128 || M % 4 != 0 || 256 % M != 0) return P24_EINVAL;
  if (cols % M != 0) return P24_EINVAL;
  P24_TRY(check_dense(A, rows, cols, lda));
  P24_TRY(check_sparse(out));
  if (out->rows != rows || out->cols != 4 * (cols / M)) return P24_EINVAL;
  if (rows > 0 && cols > 0 && !colidx) return P24_EINVAL;
  if (A_masked) {
    P24_TRY(check_dense(A_masked, rows, cols, ldam));
    if (A_masked == A && ldam != lda) return P24_EINVAL;
    if (V > 256 || cols % 8 != 0) return P24_EUNSUPPORTED;
  }
  return cuda_status(launch_vnm_compress(A, rows, cols, lda, static_cast<int>(V), static_cast<int>(M), colidx, *out,
                                         A_masked, ldam, as_stream(stream)));
}

int vnm24_spmm(const uint8_t* colidx, const p24_sparse* A, int64_t V, int64_t M, const void* B, int64_t N, int64_t ldb,
               const float* bias, uint32_t flags, void* Y, int64_t ldy, void* stream) {
  if (flags & ~(P24_EPI_BIAS | P24_EPI_RELU)) return P24_EINVAL;
  if (V < 1 || V > kMaxDim) return P24_EINVAL;
  if (M < 4 || M > 128 || M % 4 != 0 || 256 % M != 0) return P24_EINVAL;
  P24_TRY(check_sparse(A));
  const int64_t R = A->rows, Kc = A->cols;
  const int64_t K = Kc / 4 * M;
  if (K > kMaxDim || N < 0 || N > kMaxDim) return P24_EINVAL;
  P24_TRY(check_dense(B, K, N, ldb));
  P24_TRY(check_dense(Y, R, N, ldy));
  if ((flags & P24_EPI_BIAS) && !bias) return P24_EINVAL;
  if (R == 0 || N == 0) return P24_OK;
  if (!colidx) return P24_EINVAL;
  if (!aligned16(colidx)) return P24_EALIGN;
  if (Kc == 0 || V % 256 != 0 || Kc % 128 != 0 || N % 256 != 0) return P24_EUNSUPPORTED;
  int* st = device_status_ptr();
  if (!st) return P24_ECUDA;
  return cuda_status(launch_vnm_spmm(colidx, *A, static_cast<int>(V), static_cast<int>(M), B, N, ldb,
                                     (flags & P24_EPI_BIAS) ? bias : nullptr, (flags & P24_EPI_RELU) != 0, Y, ldy, st,
                                     as_stream(stream)));
}

namespace {
// the rank-r term of a low-rank call: rows of its two factors and their strides
int check_lowrank(const void* a, int64_t rows_a, int64_t lda, const void* b, int64_t rows_b, int64_t ldb, int64_t r,
                  p24::EpiArgs& epi) {
  if (r <= 0 || r % 8 != 0) return P24_EINVAL;
  P24_TRY(check_dense(a, rows_a, r, lda));
  P24_TRY(check_dense(b, rows_b, r, ldb));
  if (rows_a > 0 && rows_b > 0 && (!a || !b)) return P24_EINVAL;
  epi.lr_a = a;
  epi.lr_lda = lda;
  epi.lr_b = b;
  epi.lr_ldb = ldb;
  epi.lr_r = r;
  return P24_OK;
}

int fwd_impl(const void* X, int64_t M, int64_t ldx, const p24_sparse* W, const float* bias, uint32_t flags, void* Y,
             int64_t ldy, const p24_sparse* Y24, EpiArgs epi, void* stream) {
  if (flags & ~(P24_EPI_BIAS | P24_EPI_RELU | P24_EPI_ACT24 | P24_EPI_TEST_STALL)) return P24_EINVAL;
  epi.test_stall = (flags & P24_EPI_TEST_STALL) != 0;
  P24_TRY(check_sparse(W));
  const int64_t N = W->rows, K = W->cols;
  if (K % 8 != 0 || N % 8 != 0) return P24_EINVAL;
  P24_TRY(check_dense(X, M, K, ldx));
  P24_TRY(check_dense(Y, M, N, ldy));
  if ((flags & P24_EPI_BIAS) && !bias) return P24_EINVAL;
  epi.bias = (flags & P24_EPI_BIAS) ? bias : nullptr;
  epi.relu = (flags & P24_EPI_RELU) != 0;
  if (flags & P24_EPI_ACT24) {
    P24_TRY(check_sparse(Y24));
    if (Y24->rows != M || Y24->cols != N) return P24_EINVAL;
    epi.act24 = *Y24;
  }
  if (M == 0 || N == 0) return P24_OK;
  if (K == 0) return P24_EUNSUPPORTED;
  const cudaStream_t s = as_stream(stream);
  int* st = device_status_ptr();
  if (!st) return P24_ECUDA;
  P24_TRY(cuda_status(launch_spmm(*W, X, M, ldx, Y, ldy, /*transposed_out=*/true, epi, st, s)));
  if (flags & P24_EPI_ACT24) return cuda_status(launch_pad(*Y24, s));
  return P24_OK;
}
}  // namespace

int spmm24_fwd(const void* X, int64_t M, int64_t ldx, const p24_sparse* W, const float* bias, uint32_t flags,
               void* Y, int64_t ldy, const p24_sparse* Y24, void* stream) {
  return fwd_impl(X, M, ldx, W, bias, flags, Y, ldy, Y24, EpiArgs{}, stream);
}

int spmm24_fwd_lowrank(const void* X, int64_t M, int64_t ldx, const p24_sparse* W, const void* T, int64_t ldt,
                       const void* L, int64_t ldl, int64_t r, const float* bias, uint32_t flags, void* Y, int64_t ldy,
                       const p24_sparse* Y24, void* stream) {
  P24_TRY(check_sparse(W));
  EpiArgs epi;
  P24_TRY(check_lowrank(L, W->rows, ldl, T, M, ldt, r, epi));
  return fwd_impl(X, M, ldx, W, bias, flags, Y, ldy, Y24, epi, stream);
}

int spmm24_fwd_sparse_act(const p24_sparse* Xs, const void* Wm, int64_t N, int64_t ldw, const float* bias,
                          uint32_t flags, void* Y, int64_t ldy, void* stream) {
  if (flags & ~(P24_EPI_BIAS | P24_EPI_RELU)) return P24_EINVAL;
  P24_TRY(check_sparse(Xs));
  const int64_t M = Xs->rows, K = Xs->cols;
  if (K % 8 != 0 || N % 8 != 0) return P24_EINVAL;
  P24_TRY(check_dense(Wm, N, K, ldw));
  P24_TRY(check_dense(Y, M, N, ldy));
  if ((flags & P24_EPI_BIAS) && !bias) return P24_EINVAL;
  if (M == 0 || N == 0) return P24_OK;
  if (K == 0) return P24_EUNSUPPORTED;
  EpiArgs epi;
  epi.bias = (flags & P24_EPI_BIAS) ? bias : nullptr;
  epi.relu = (flags & P24_EPI_RELU) != 0;
  int* st = device_status_ptr();
  if (!st) return P24_ECUDA;
  return cuda_status(launch_spmm(*Xs, Wm, N, ldw, Y, ldy, /*transposed_out=*/false, epi, st, as_stream(stream)));
}

namespace {
int bwd_dx_impl(const void* dY, int64_t M, int64_t lddy, const p24_sparse* WbwdT, const void* gate, int64_t ldg,
                void* dX, int64_t lddx, float* dbias, EpiArgs epi, void* stream) {
  P24_TRY(check_sparse(WbwdT));
  const int64_t K = WbwdT->rows, N = WbwdT->cols;
  if (K % 8 != 0 || N % 8 != 0) return P24_EINVAL;
  P24_TRY(check_dense(dY, M, N, lddy));
  P24_TRY(check_dense(dX, M, K, lddx));
  if (gate) P24_TRY(check_dense(gate, M, K, ldg));
  if (dbias && !aligned16(dbias)) return P24_EALIGN;
  if (K == 0) return P24_OK;
  if (dbias) P24_TRY(cuda_status(cudaMemsetAsync(dbias, 0, K * 4, as_stream(stream))));
  if (M == 0) return P24_OK;
  if (N == 0) return P24_EUNSUPPORTED;
  epi.gate = gate;
  epi.ldg = ldg;
  epi.dbias = dbias;
  int* st = device_status_ptr();
  if (!st) return P24_ECUDA;
  return cuda_status(launch_spmm(*WbwdT, dY, M, lddy, dX, lddx, /*transposed_out=*/true, epi, st, as_stream(stream)));
}
}  // namespace

int spmm24_bwd_dx(const void* dY, int64_t M, int64_t lddy, const p24_sparse* WbwdT, const void* gate, int64_t ldg,
                  void* dX, int64_t lddx, float* dbias, void* stream) {
  return bwd_dx_impl(dY, M, lddy, WbwdT, gate, ldg, dX, lddx, dbias, EpiArgs{}, stream);
}

int spmm24_bwd_dx_lowrank(const void* dY, int64_t M, int64_t lddy, const p24_sparse* WbwdT, const void* U,
                          int64_t ldu, const void* Rt, int64_t ldrt, int64_t r, const void* gate, int64_t ldg, void* dX,
                          int64_t lddx, float* dbias, void* stream) {
  P24_TRY(check_sparse(WbwdT));
  EpiArgs epi;
  P24_TRY(check_lowrank(Rt, WbwdT->rows, ldrt, U, M, ldu, r, epi));
  return bwd_dx_impl(dY, M, lddy, WbwdT, gate, ldg, dX, lddx, dbias, epi, stream);
}

int p24_gemm_nt(const void* A, int64_t M, int64_t lda, const void* B, int64_t N, int64_t ldb, int64_t K, void* C,
                int64_t ldc, void* stream) {
  if (K < 0) return P24_EINVAL;
  P24_TRY(check_dense(A, M, K, lda));
  P24_TRY(check_dense(B, N, K, ldb));
  P24_TRY(check_dense(C, M, N, ldc));
  int* st = device_status_ptr();
  if (!st) return P24_ECUDA;
  return cuda_status(launch_gemm_nt(A, M, lda, B, N, ldb, K, C, ldc, st, as_stream(stream)));
}

int p24_gemm_tn(const void* A, int64_t lda, const void* B, int64_t ldb, int64_t M, int64_t N, int64_t K, void* C,
                int64_t ldc, void* stream) {
  P24_TRY(check_dense(A, M, N, lda));
  P24_TRY(check_dense(B, M, K, ldb));
  P24_TRY(check_dense(C, N, K, ldc));
  int* st = device_status_ptr();
  if (!st) return P24_ECUDA;
  return cuda_status(launch_gemm_tn(A, lda, B, ldb, M, N, K, C, ldc, st, as_stream(stream)));
}

int p24_transpose(const void* src, int64_t rows, int64_t cols, int64_t lds, void* dst, int64_t ldd, void* stream) {
  // element-wise accesses: any stride and 2-byte alignment will do
  if (rows < 0 || cols < 0 || rows > kMaxDim || cols > kMaxDim) return P24_EINVAL;
  if (rows == 0 || cols == 0) return P24_OK;
  if (!src || !dst || lds < cols || ldd < rows) return P24_EINVAL;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 1) return P24_EALIGN;
  return cuda_status(launch_transpose_bf16(src, rows, cols, lds, dst, ldd, as_stream(stream)));
}

int masked_dw_gemm(const void* dY, int64_t lddy, const void* X, int64_t ldx, int64_t M, const p24_sparse* Wfwd,
                   void* dW, int64_t lddw, void* stream) {
  P24_TRY(check_sparse(Wfwd));
  const int64_t N = Wfwd->rows, K = Wfwd->cols;
  if (K % 8 != 0 || N % 8 != 0) return P24_EINVAL;
  P24_TRY(check_dense(dY, M, N, lddy));
  P24_TRY(check_dense(X, M, K, ldx));
  P24_TRY(check_dense(dW, N, K, lddw));
  int* st = device_status_ptr();
  if (!st) return P24_ECUDA;
  return cuda_status(
      launch_masked_dw(dY, lddy, X, ldx, M, N, K, Wfwd->meta, Wfwd->ldm, dW, lddw, st, as_stream(stream)));
}

size_t p24_colsum_workspace_size(int64_t M, int64_t N) {
  if (M < 0 || N < 0) return 0;
  return static_cast<size_t>(colsum_slabs(M) * N * 4);
}

int p24_colsum(const void* G, int64_t M, int64_t N, int64_t ldg, float* out, void* ws, size_t ws_bytes,
               void* stream) {
  P24_TRY(check_dense(G, M, N, ldg));
  if (N > 0 && !out) return P24_EINVAL;
  if (N > 0 && !aligned16(out)) return P24_EALIGN;
  if (N > 0 && M > 0) {
    if (!ws) return P24_EINVAL;
    if (!aligned16(ws)) return P24_EALIGN;
    if (ws_bytes < p24_colsum_workspace_size(M, N)) return P24_ENOSPACE;
  }
  return cuda_status(launch_colsum(G, M, N, ldg, out, static_cast<float*>(ws), as_stream(stream)));
}

int p24_colsum_noalloc(const void* G, int64_t M, int64_t N, int64_t ldg, float* out, void* stream) {
  P24_TRY(check_dense(G, M, N, ldg));
  if (N > 0 && !out) return P24_EINVAL;
  if (N > 0 && !aligned16(out)) return P24_EALIGN;
  if (N > P24_COLSUM_NOALLOC_MAX_COLS) return P24_ENOSPACE;
  return cuda_status(launch_colsum_noalloc(G, M, N, ldg, out, as_stream(stream)));
}

size_t ffn24_workspace_size_lowrank(int64_t M, int64_t d, int64_t ffn, uint32_t flags, int64_t r) {
  if (M < 0 || d < 0 || ffn < 0 || r < 0) return 0;
  StepLayout L;
  void *wdm, *dH;
  float* cs;
  step_layout(M, d, ffn, flags, r, nullptr, L, &wdm, &dH, &cs);
  return L.total;
}

size_t ffn24_workspace_size(int64_t M, int64_t d, int64_t ffn, uint32_t flags) {
  return ffn24_workspace_size_lowrank(M, d, ffn, flags, 0);
}

size_t ffn24_workspace_size_args(const p24_ffn_args* a) {
  if (!a || a->M < 0 || a->d < 0 || a->ffn < 0 || a->r < 0) return 0;
  const bool vnm = (a->flags & P24_STEP_VNM) != 0;
  if (vnm && (a->vnm_V <= 0 || a->vnm_M < 4 || a->vnm_M % 4 != 0 || a->ffn % a->vnm_M != 0)) return 0;
  StepLayout L;
  void *wdm, *dH;
  float* cs;
  step_layout(a->M, a->d, a->ffn, a->flags, (a->flags & P24_STEP_ADAPTERS) ? a->r : 0, nullptr, L, &wdm, &dH, &cs,
              vnm ? a->vnm_V : 0, vnm ? a->vnm_M : 0);
  return L.total;
}

int ffn24_step(const p24_ffn_args* a, void* workspace, size_t ws_bytes, void* stream) {
  return ffn24_step_traced(a, workspace, ws_bytes, stream, nullptr, 0);
}

uint64_t p24_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int ffn24_step_traced(const p24_ffn_args* a, void* workspace, size_t ws_bytes, void* stream, void* const* events,
                      int n_events) {
  if (!a) return P24_EINVAL;
  if (n_events < 0 || (n_events > 0 && !events)) return P24_EINVAL;
  if (a->flags & ~(P24_STEP_ACT24 | P24_STEP_KEEP_MASKS | P24_STEP_ADAPTERS | P24_STEP_VNM)) return P24_EINVAL;
  const int64_t M = a->M, d = a->d, ffn = a->ffn;
  if (M < 0 || d <= 0 || ffn <= 0 || d % 8 != 0 || ffn % 8 != 0) return P24_EINVAL;
  const bool act24 = (a->flags & P24_STEP_ACT24) != 0;
  const bool vnm = (a->flags & P24_STEP_VNM) != 0;
  const int64_t vV = vnm ? a->vnm_V : 0, vM = vnm ? a->vnm_M : 0;
  if (vnm) {
    if (vM < 4 || vM > 128 || vM % 4 != 0 || 256 % vM != 0 || vV < 1) return P24_EINVAL;
    if (act24 || (a->flags & P24_STEP_ADAPTERS)) return P24_EUNSUPPORTED;
    if (vV != 256 || ffn % (32 * vM) != 0 || d % 256 != 0) return P24_EUNSUPPORTED;
  }
  const bool keep = (a->flags & P24_STEP_KEEP_MASKS) != 0;
  // caller's compressed weights: required with fixed masks, optional otherwise
  const p24_sparse* cw[4] = {a->up_fwd, a->up_bwdT, a->down_fwd, a->down_bwdT};
  const int64_t cw_rows[4] = {ffn, d, d, ffn}, cw_cols[4] = {d, ffn, ffn, d};
  for (int i = 0; i < 4; ++i) {
    if (!cw[i]) {
      if (keep) return P24_EINVAL;
      continue;
    }
    P24_TRY(check_sparse(cw[i]));
    if (cw[i]->rows != cw_rows[i] || cw[i]->cols != cw_cols[i]) return P24_EINVAL;
  }
  if (keep && act24 && !a->W_down_masked) return P24_EINVAL;
  if (a->W_down_masked) P24_TRY(check_dense(a->W_down_masked, d, ffn, ffn));
  if (a->dH) P24_TRY(check_dense(a->dH, M, ffn, ffn));
  const bool ad = (a->flags & P24_STEP_ADAPTERS) != 0;
  const int64_t r = a->r;
  if (ad) {
    if (r <= 0 || r % 8 != 0) return P24_EINVAL;
    const void* in[4] = {a->L_up, a->R_up, a->L_down, a->R_down};
    const void* out[4] = {a->dL_up, a->dR_up, a->dL_down, a->dR_down};
    const int64_t rows[4] = {ffn, r, d, r}, cols[4] = {r, d, r, ffn};
    for (int i = 0; i < 4; ++i) {
      if (!in[i] || !out[i]) return P24_EINVAL;
      P24_TRY(check_dense(in[i], rows[i], cols[i], cols[i]));
      P24_TRY(check_dense(out[i], rows[i], cols[i], cols[i]));
    }
  }
  if (!keep) {
    P24_TRY(check_dense(a->W_up, ffn, d, d));
    P24_TRY(check_dense(a->W_down, d, ffn, ffn));
  }
  P24_TRY(check_dense(a->dW_up, ffn, d, d));
  P24_TRY(check_dense(a->dW_down, d, ffn, ffn));
  if (M > 0) {
    P24_TRY(check_dense(a->X, M, d, d));
    P24_TRY(check_dense(a->dY, M, d, d));
    P24_TRY(check_dense(a->Y, M, d, d));
    P24_TRY(check_dense(a->dX, M, d, d));
    P24_TRY(check_dense(a->H, M, ffn, ffn));
  }
  for (const void* p : {static_cast<const void*>(a->b_up), static_cast<const void*>(a->b_down),
                        static_cast<const void*>(a->db_up), static_cast<const void*>(a->db_down)})
    if (p && !aligned16(p)) return P24_EALIGN;
  if (!workspace) return P24_EINVAL;
  if (!aligned16(workspace)) return P24_EALIGN;
  StepLayout L;
  void *wdm, *dHv;
  float* cs;
  step_layout(M, d, ffn, a->flags, ad ? r : 0, static_cast<char*>(workspace), L, &wdm, &dHv, &cs, vV, vM);
  if (ws_bytes < L.total) return P24_ENOSPACE;
  const cudaStream_t s = as_stream(stream);
  int* st = device_status_ptr();
  if (!st) return P24_ECUDA;
  const int n_ph = n_events / 2 < P24_STEP_PHASES ? n_events / 2 : P24_STEP_PHASES;
  auto mark = [&](int phase, int edge) -> int {
    if (phase >= n_ph) return P24_OK;
    return cuda_status(cudaEventRecord(static_cast<cudaEvent_t>(events[2 * phase + edge]), s));
  };
#define P24_PHASE(ph, body)   \
  do {                        \
    P24_TRY(mark(ph, 0));     \
    body;                     \
    P24_TRY(mark(ph, 1));     \
  } while (0)

  // caller buffers replace the workspace's copies
  const p24_sparse ws_dn_bwdT = L.dn_bwdT;
  if (a->up_fwd) L.up_fwd = *a->up_fwd;
  if (a->up_bwdT) L.up_bwdT = *a->up_bwdT;
  if (a->down_fwd) L.dn_fwd = *a->down_fwd;
  if (a->down_bwdT) L.dn_bwdT = *a->down_bwdT;
  if (a->W_down_masked) wdm = a->W_down_masked;
  if (a->dH) dHv = a->dH;
  // 1. fresh 2:4 masks of both weights, and their double-pruned transposes (GMP);
  //    with fixed masks the caller's compressed weights are used as they are
  //    (with adapters, also the transposed factors their backward products need)
  P24_PHASE(0, {
    if (!keep) P24_TRY(cuda_status(launch_compress_both(a->W_up, ffn, d, d, L.up_fwd, L.up_bwdT, nullptr, 0, s)));
    if (ad) {
      P24_TRY(cuda_status(launch_transpose_bf16(a->L_up, ffn, r, r, L.Lt_up, ffn, s)));
      P24_TRY(cuda_status(launch_transpose_bf16(a->R_up, r, d, d, L.Rt_up, r, s)));
    }
  });
  P24_PHASE(1, {
    if (vnm) {
      // W_down on its mask, transposed [ffn, d]: the gathered operand of the V:2:M down GEMM
      // (a caller's W_down_masked, if any, is written by a plain compress beside it)
      if (!keep) {
        P24_TRY(cuda_status(launch_compress_both(a->W_down, d, ffn, ffn, L.dn_fwd, L.dn_bwdT, nullptr, 0, s,
                                                 L.wdmT, d)));
        // the caller's row-major W_down on its mask, if asked for (the forward prune again)
        if (a->W_down_masked)
          P24_TRY(cuda_status(launch_compress(a->W_down, d, ffn, ffn, L.dn_fwd, a->W_down_masked, ffn, s)));
      } else {
        // fixed masks: from the caller's compressed W_down; its double prune goes to the
        // workspace's copy (the caller's buffers are read only)
        P24_TRY(cuda_status(launch_transpose_repack(L.dn_fwd, ws_dn_bwdT, s, L.wdmT, d)));
      }
    } else if (!keep) {
      P24_TRY(cuda_status(launch_compress_both(a->W_down, d, ffn, ffn, L.dn_fwd, L.dn_bwdT,
                                               (act24 || a->W_down_masked) ? wdm : nullptr, ffn, s)));
    }
    if (ad) {
      P24_TRY(cuda_status(launch_transpose_bf16(a->L_down, d, r, r, L.Lt_dn, d, s)));
      P24_TRY(cuda_status(launch_transpose_bf16(a->R_down, r, ffn, ffn, L.Rt_dn, r, s)));
    }
  });
  if (M == 0) {
    if (ad) {  // empty sums: zero adapter gradients
      P24_TRY(cuda_status(cudaMemsetAsync(a->dL_up, 0, ffn * r * 2, s)));
      P24_TRY(cuda_status(cudaMemsetAsync(a->dR_up, 0, r * d * 2, s)));
      P24_TRY(cuda_status(cudaMemsetAsync(a->dL_down, 0, d * r * 2, s)));
      P24_TRY(cuda_status(cudaMemsetAsync(a->dR_down, 0, r * ffn * 2, s)));
    }
    if (a->db_up) P24_TRY(cuda_status(cudaMemsetAsync(a->db_up, 0, ffn * 4, s)));
    if (a->db_down) P24_TRY(cuda_status(cudaMemsetAsync(a->db_down, 0, d * 4, s)));
    P24_TRY(cuda_status(cudaMemsetAsync(a->dW_up, 0, ffn * d * 2, s)));
    return cuda_status(cudaMemsetAsync(a->dW_down, 0, ffn * d * 2, s));
  }
  // 2. H = ReLU(X W_up^T + b_up)  [ACT24: pruned 2:4 along ffn, compressed copy in hs]
  EpiArgs up;
  up.bias = a->b_up;
  up.relu = true;
  if (act24) up.act24 = L.hs;
  if (ad) {  // + T_up L_up^T, T_up = X R_up^T
    up.lr_a = a->L_up, up.lr_lda = r, up.lr_b = L.T_up, up.lr_ldb = r, up.lr_r = r;
  }
  P24_PHASE(2, {
    if (ad) P24_TRY(cuda_status(launch_gemm_nt(a->X, M, d, a->R_up, r, d, d, L.T_up, r, st, s)));
    P24_TRY(cuda_status(launch_spmm(L.up_fwd, a->X, M, d, a->H, ffn, true, up, st, s)));
    if (act24) P24_TRY(cuda_status(launch_pad(L.hs, s)));
    // V:N:M: prune H V:2:M along ffn, in place, and keep its condensed form for the down GEMM
    if (vnm)
      P24_TRY(cuda_status(launch_vnm_compress(a->H, M, ffn, ffn, static_cast<int>(vV), static_cast<int>(vM),
                                              L.colidx, L.hs, a->H, ffn, s)));
  });
  // 3. Y = H W_down^T + b_down
  EpiArgs dn;
  dn.bias = a->b_down;
  if (ad) {  // + T_dn L_down^T, T_dn = H R_down^T (A and B swap roles in the sparse-activation form)
    dn.lr_r = r;
    if (act24) dn.lr_a = L.T_dn, dn.lr_lda = r, dn.lr_b = a->L_down, dn.lr_ldb = r;
    else dn.lr_a = a->L_down, dn.lr_lda = r, dn.lr_b = L.T_dn, dn.lr_ldb = r;
  }
  P24_PHASE(3, {
    if (ad) P24_TRY(cuda_status(launch_gemm_nt(a->H, M, ffn, a->R_down, r, ffn, ffn, L.T_dn, r, st, s)));
    if (act24) P24_TRY(cuda_status(launch_spmm(L.hs, wdm, d, ffn, a->Y, d, false, dn, st, s)));
    else if (vnm)
      P24_TRY(cuda_status(launch_vnm_spmm(L.colidx, L.hs, static_cast<int>(vV), static_cast<int>(vM), L.wdmT, d, d,
                                          a->b_down, false, a->Y, d, st, s)));
    else P24_TRY(cuda_status(launch_spmm(L.dn_fwd, a->H, M, ffn, a->Y, d, true, dn, st, s)));
  });
  // 4. dH = (dY W_down_bwd) * [H > 0], with db_up = column sums of dH fused into its epilogue
  EpiArgs g;
  g.gate = a->H;
  g.ldg = ffn;
  g.dbias = a->db_up;
  if (ad) {  // + U_dn R_down, U_dn = dY L_down
    g.lr_a = L.Rt_dn, g.lr_lda = r, g.lr_b = L.U_dn, g.lr_ldb = r, g.lr_r = r;
  }
  P24_PHASE(4, {
    if (ad) P24_TRY(cuda_status(launch_gemm_nt(a->dY, M, d, L.Lt_dn, r, d, d, L.U_dn, r, st, s)));
    if (a->db_up) P24_TRY(cuda_status(cudaMemsetAsync(a->db_up, 0, ffn * 4, s)));
    P24_TRY(cuda_status(launch_spmm(L.dn_bwdT, a->dY, M, d, dHv, ffn, true, g, st, s)));
  });
  // 5. db_down = column sums of dY
  P24_PHASE(5, {
    if (a->db_down) P24_TRY(cuda_status(launch_colsum_step(a->dY, M, d, d, a->db_down, cs, s)));
  });
  // 6. dW_down = (dY^T H) on mask(W_down)
  P24_PHASE(6, {
    if (ad) {  // dR_down = U_dn^T H as extra rows of the same pass over H; dL_down = dY^T T_dn
      DwExtra ex;
      ex.a2 = L.U_dn;
      ex.lda2 = r;
      ex.n2 = r;
      ex.out2 = a->dR_down;
      ex.ldo2 = ffn;
      P24_TRY(cuda_status(launch_masked_dw_extra(a->dY, d, a->H, ffn, M, d, ffn, L.dn_fwd.meta, L.dn_fwd.ldm,
                                                 a->dW_down, ffn, ex, st, s)));
      P24_TRY(cuda_status(launch_gemm_tn(a->dY, d, L.T_dn, r, M, d, r, a->dL_down, r, st, s)));
    } else {
      P24_TRY(cuda_status(launch_masked_dw(a->dY, d, a->H, ffn, M, d, ffn, L.dn_fwd.meta, L.dn_fwd.ldm, a->dW_down,
                                           ffn, st, s)));
    }
  });
  // 7. dX = dH W_up_bwd
  EpiArgs gx;
  if (ad) {  // + U_up R_up, U_up = dH L_up
    gx.lr_a = L.Rt_up, gx.lr_lda = r, gx.lr_b = L.U_up, gx.lr_ldb = r, gx.lr_r = r;
  }
  P24_PHASE(7, {
    if (ad) P24_TRY(cuda_status(launch_gemm_nt(dHv, M, ffn, L.Lt_up, r, ffn, ffn, L.U_up, r, st, s)));
    P24_TRY(cuda_status(launch_spmm(L.up_bwdT, dHv, M, ffn, a->dX, d, true, gx, st, s)));
  });
  // 8. dW_up = (dH^T X) on mask(W_up)
  P24_PHASE(8, {
    if (ad) {  // dL_up = dH^T T_up as extra columns of the same pass over dH; dR_up = U_up^T X
      DwExtra ex;
      ex.b2 = L.T_up;
      ex.ldb2 = r;
      ex.k2 = r;
      ex.out2 = a->dL_up;
      ex.ldo2 = r;
      P24_TRY(cuda_status(launch_masked_dw_extra(dHv, ffn, a->X, d, M, ffn, d, L.up_fwd.meta, L.up_fwd.ldm,
                                                 a->dW_up, d, ex, st, s)));
      P24_TRY(cuda_status(launch_gemm_tn(L.U_up, r, a->X, d, M, r, d, a->dR_up, d, st, s)));
    } else {
      P24_TRY(cuda_status(
          launch_masked_dw(dHv, ffn, a->X, d, M, ffn, d, L.up_fwd.meta, L.up_fwd.ldm, a->dW_up, d, st, s)));
    }
  });
#undef P24_PHASE
  return P24_OK;
}

namespace {
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int check_hybrid(const p24_hybrid* h) {
  if (!h) return P24_EINVAL;
  if (h->rows < 0 || h->rows > kMaxDim || h->cols < 0 || h->cols > 65536 || h->E < 1 || h->E > kMaxDim ||
      h->cap < 0 || h->cap > kMaxDim)
    return P24_EINVAL;
  if (h->cols % 8 != 0) return P24_EINVAL;
  if (h->rows == 0) return P24_OK;
  if (!h->nnz || !h->ell_cols || !h->ell_vals || !h->slot || !h->n_ovf) return P24_EINVAL;
  if (h->cap > 0 && (!h->ovf_rows || !h->ovf)) return P24_EINVAL;
  if (!aligned4(h->nnz) || !aligned4(h->slot) || !aligned4(h->n_ovf) || (h->cap > 0 && !aligned4(h->ovf_rows)))
    return P24_EALIGN;
  if (!aligned16(h->ell_cols) || !aligned16(h->ell_vals)) return P24_EALIGN;
  if (h->cap > 0) P24_TRY(check_dense(h->ovf, h->cap, h->cols, h->ldo));
  return P24_OK;
}
}  // namespace

int hyb_compress(const void* A, int64_t lda, const p24_hybrid* h, void* stream) {
  P24_TRY(check_hybrid(h));
  P24_TRY(check_dense(A, h->rows, h->cols, lda));
  if (h->rows == 0) return P24_OK;
  int* st = device_status_ptr();
  if (!st) return P24_ECUDA;
  return cuda_status(launch_hyb_compress(A, lda, *h, st, as_stream(stream)));
}

int hyb_spmm(const p24_hybrid* h, const void* B, int64_t N, int64_t ldb, void* Y, int64_t ldy, void* stream) {
  P24_TRY(check_hybrid(h));
  if (N < 0 || N > kMaxDim || N % 8 != 0) return P24_EINVAL;
  P24_TRY(check_dense(B, h->cols, N, ldb));
  P24_TRY(check_dense(Y, h->rows, N, ldy));
  if (h->rows == 0 || N == 0) return P24_OK;
  return cuda_status(launch_hyb_spmm(*h, B, N, ldb, Y, ldy, as_stream(stream)));
}

int hyb_sddmm(const p24_hybrid* h, const void* G, int64_t N, int64_t ldg, const void* B, int64_t ldb, void* S_ell,
              void* S_ovf, int64_t lds, void* stream) {
  P24_TRY(check_hybrid(h));
  if (N < 0 || N > 32768 || N % 8 != 0) return P24_EINVAL;  // G's row is staged in shared memory
  P24_TRY(check_dense(G, h->rows, N, ldg));
  P24_TRY(check_dense(B, h->cols, N, ldb));
  if (h->rows > 0 && (!S_ell || !aligned16(S_ell))) return S_ell ? P24_EALIGN : P24_EINVAL;
  if (h->cap > 0) P24_TRY(check_dense(S_ovf, h->cap, h->cols, lds));
  if (h->rows == 0) return P24_OK;
  return cuda_status(launch_hyb_sddmm(*h, G, N, ldg, B, ldb, S_ell, S_ovf, lds, as_stream(stream)));
}

int p24_selftest_timeout(int64_t limit_ns, void* stream) {
  if (limit_ns <= 0 || limit_ns > 10000000000LL) return P24_EINVAL;
  int* st = device_status_ptr();
  if (!st) return P24_ECUDA;
  return cuda_status(launch_selftest_timeout(static_cast<uint64_t>(limit_ns), st, as_stream(stream)));
}

int p24_query_timeout(void* stream, int64_t* cta, int64_t* barrier) {
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return P24_ECUDA;
  int v[4] = {0, 0, 0, 0};
  if (cudaMemcpyFromSymbol(v, g_status, sizeof(v)) != cudaSuccess) return P24_ECUDA;
  const int zero[4] = {0, 0, 0, 0};
  if (cudaMemcpyToSymbol(g_status, zero, sizeof(zero)) != cudaSuccess) return P24_ECUDA;
  if (cta) *cta = v[0] ? static_cast<int64_t>(v[1]) : int64_t(-1);
  if (barrier) *barrier = v[0] ? static_cast<int64_t>(static_cast<uint32_t>(v[2])) : int64_t(-1);
  return v[0];
}

int p24_query_status(void* stream) { return p24_query_timeout(stream, nullptr, nullptr); }

const char* p24_strerror(int code) {
  switch (code) {
    case P24_OK: return "ok";
    case P24_EINVAL: return "invalid argument (null pointer, shape or flag)";
    case P24_EALIGN: return "pointer or row stride not 16-byte aligned";
    case P24_ECUDA: return "CUDA call or kernel launch failed";
    case P24_ETIMEOUT: return "a kernel's bounded wait expired";
    case P24_EUNSUPPORTED: return "unsupported device or shape";
    case P24_ENOSPACE: return "workspace too small";
    case P24_ECAPACITY: return "a data-dependent output exceeded its capacity";
    default: return "unknown status";
  }
}

}  // extern "C"
