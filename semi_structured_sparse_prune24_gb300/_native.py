"""ctypes binding of libprune24 (include/prune24.h): argument marshalling only.

Every call forwards raw device pointers, sizes and row strides of torch tensors
to the C ABI and runs on the current torch CUDA stream; all arithmetic happens
in the library's CUDA kernels. Output tensors the caller does not pass are
allocated with torch (device memory is torch's job here). There is no CPU path:
if the shared library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libprune24.so")

P24_OK, P24_EINVAL, P24_EALIGN, P24_ECUDA, P24_ETIMEOUT, P24_EUNSUPPORTED, P24_ENOSPACE = 0, -1, -2, -3, -4, -5, -6
P24_ECAPACITY = -7
P24_EPI_BIAS, P24_EPI_RELU, P24_EPI_ACT24 = 0x1, 0x2, 0x4
P24_EPI_TEST_STALL = 0x80000000
P24_STEP_ACT24 = 0x1
P24_STEP_KEEP_MASKS = 0x2
P24_STEP_ADAPTERS = 0x4
P24_STEP_VNM = 0x8


class P24Error(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {lib.p24_strerror(code).decode()} (status {code})")


class p24_sparse(C.Structure):
    _fields_ = [("vals", C.c_void_p), ("meta", C.c_void_p), ("rows", C.c_int64), ("cols", C.c_int64),
                ("ldv", C.c_int64), ("ldm", C.c_int64)]


class p24_ffn_args(C.Structure):
    _fields_ = [("M", C.c_int64), ("d", C.c_int64), ("ffn", C.c_int64), ("flags", C.c_uint32),
                ("X", C.c_void_p), ("W_up", C.c_void_p), ("b_up", C.c_void_p), ("W_down", C.c_void_p),
                ("b_down", C.c_void_p), ("dY", C.c_void_p), ("Y", C.c_void_p), ("H", C.c_void_p),
                ("dX", C.c_void_p), ("dW_up", C.c_void_p), ("dW_down", C.c_void_p), ("db_up", C.c_void_p),
                ("db_down", C.c_void_p), ("up_fwd", C.POINTER(p24_sparse)), ("up_bwdT", C.POINTER(p24_sparse)),
                ("down_fwd", C.POINTER(p24_sparse)), ("down_bwdT", C.POINTER(p24_sparse)),
                ("W_down_masked", C.c_void_p), ("r", C.c_int64), ("L_up", C.c_void_p), ("R_up", C.c_void_p),
                ("L_down", C.c_void_p), ("R_down", C.c_void_p), ("dL_up", C.c_void_p), ("dR_up", C.c_void_p),
                ("dL_down", C.c_void_p), ("dR_down", C.c_void_p), ("dH", C.c_void_p), ("vnm_V", C.c_int64),
                ("vnm_M", C.c_int64)]


class p24_hybrid(C.Structure):
    _fields_ = [("rows", C.c_int64), ("cols", C.c_int64), ("E", C.c_int64), ("cap", C.c_int64),
                ("nnz", C.c_void_p), ("ell_cols", C.c_void_p), ("ell_vals", C.c_void_p), ("slot", C.c_void_p),
                ("ovf_rows", C.c_void_p), ("n_ovf", C.c_void_p), ("ovf", C.c_void_p), ("ldo", C.c_int64)]


def _load() -> C.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libprune24 is not built ({_LIB_PATH} missing): run __graft_entry__.build() "
                          "or python semi_structured_sparse_prune24_gb300/build.py")
    L = C.CDLL(_LIB_PATH)
    i64, vp, u32, sz, i32 = C.c_int64, C.c_void_p, C.c_uint32, C.c_size_t, C.c_int
    sp = C.POINTER(p24_sparse)
    sigs = {
        "p24_ld_vals": (i64, [i64]),
        "p24_ld_meta": (i64, [i64]),
        "prune24_compress": (i32, [vp, i64, i64, i64, sp, vp, i64, vp]),
        "prune24_transpose_repack": (i32, [sp, sp, vp]),
        "prune24_compress_both": (i32, [vp, i64, i64, i64, sp, sp, vp, i64, vp]),
        "vnm24_compress": (i32, [vp, i64, i64, i64, i64, i64, vp, sp, vp, i64, vp]),
        "vnm24_spmm": (i32, [vp, sp, i64, i64, vp, i64, i64, vp, u32, vp, i64, vp]),
        "spmm24_fwd": (i32, [vp, i64, i64, sp, vp, u32, vp, i64, sp, vp]),
        "spmm24_fwd_sparse_act": (i32, [sp, vp, i64, i64, vp, u32, vp, i64, vp]),
        "spmm24_bwd_dx": (i32, [vp, i64, i64, sp, vp, i64, vp, i64, vp, vp]),
        "masked_dw_gemm": (i32, [vp, i64, vp, i64, i64, sp, vp, i64, vp]),
        "spmm24_fwd_lowrank": (i32, [vp, i64, i64, sp, vp, i64, vp, i64, i64, vp, u32, vp, i64, sp, vp]),
        "spmm24_bwd_dx_lowrank": (i32, [vp, i64, i64, sp, vp, i64, vp, i64, i64, vp, i64, vp, i64, vp, vp]),
        "p24_gemm_nt": (i32, [vp, i64, i64, vp, i64, i64, i64, vp, i64, vp]),
        "p24_gemm_tn": (i32, [vp, i64, vp, i64, i64, i64, i64, vp, i64, vp]),
        "p24_transpose": (i32, [vp, i64, i64, i64, vp, i64, vp]),
        "p24_colsum_workspace_size": (sz, [i64, i64]),
        "p24_colsum": (i32, [vp, i64, i64, i64, vp, vp, sz, vp]),
        "p24_colsum_noalloc": (i32, [vp, i64, i64, i64, vp, vp]),
        "ffn24_workspace_size": (sz, [i64, i64, i64, u32]),
        "ffn24_workspace_size_lowrank": (sz, [i64, i64, i64, u32, i64]),
        "ffn24_workspace_size_args": (sz, [C.POINTER(p24_ffn_args)]),
        "ffn24_step": (i32, [C.POINTER(p24_ffn_args), vp, sz, vp]),
        "ffn24_step_traced": (i32, [C.POINTER(p24_ffn_args), vp, sz, vp, C.POINTER(vp), i32]),
        "hyb_compress": (i32, [vp, i64, C.POINTER(p24_hybrid), vp]),
        "hyb_spmm": (i32, [C.POINTER(p24_hybrid), vp, i64, i64, vp, i64, vp]),
        "hyb_sddmm": (i32, [C.POINTER(p24_hybrid), vp, i64, i64, vp, i64, vp, vp, i64, vp]),
        "p24_launch_count": (C.c_uint64, []),
        "p24_query_status": (i32, [vp]),
        "p24_query_timeout": (i32, [vp, C.POINTER(i64), C.POINTER(i64)]),
        "p24_selftest_timeout": (i32, [i64, vp]),
        "p24_strerror": (C.c_char_p, [i32]),
    }
    for name, (res, args) in sigs.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


lib = _load()


def _check(code: int, where: str) -> None:
    if code != P24_OK:
        raise P24Error(code, where)


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _mat(t: torch.Tensor, dtype=torch.bfloat16, name="tensor") -> tuple[int, int, int]:
    """(rows, cols, row stride) of a row-major matrix view on a CUDA device."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libprune24 has no CPU path)")
    if t.numel() and t.stride(1) != 1:
        raise ValueError(f"{name} must be contiguous along its last dimension")
    return t.shape[0], t.shape[1], (t.stride(0) if t.shape[0] > 1 else max(t.shape[1], t.stride(0)))


def ld_vals(cols: int) -> int:
    return int(lib.p24_ld_vals(cols))


def ld_meta(cols: int) -> int:
    return int(lib.p24_ld_meta(cols))


@dataclass
class Sparse24:
    """A matrix pruned 2:4 along its columns, compressed (see p24_sparse in include/prune24.h).

    vals: bf16 [rows, ldv] (torch tensor, may be a view with row stride ldv)
    meta: uint8 [rows, ldm]
    """
    vals: torch.Tensor
    meta: torch.Tensor
    rows: int
    cols: int

    @staticmethod
    def empty(rows: int, cols: int, device="cuda", ldv: int | None = None, ldm: int | None = None) -> "Sparse24":
        ldv = ld_vals(cols) if ldv is None else ldv
        ldm = ld_meta(cols) if ldm is None else ldm
        vals = torch.empty((rows, ldv), dtype=torch.bfloat16, device=device)
        meta = torch.empty((rows, ldm), dtype=torch.uint8, device=device)
        return Sparse24(vals, meta, rows, cols)

    @property
    def ldv(self) -> int:
        return self.vals.stride(0) if self.rows > 1 else self.vals.shape[1]

    @property
    def ldm(self) -> int:
        return self.meta.stride(0) if self.rows > 1 else self.meta.shape[1]

    def c(self) -> p24_sparse:
        for t, name in ((self.vals, "vals"), (self.meta, "meta")):
            if not t.is_cuda:
                raise ValueError(f"Sparse24.{name} must be on a CUDA device")
        return p24_sparse(self.vals.data_ptr(), self.meta.data_ptr(), self.rows, self.cols, self.ldv, self.ldm)


# ------------------------------------------------------------------ entry points
def prune24_compress(W: torch.Tensor, out: Sparse24 | None = None, W_masked: torch.Tensor | None = None,
                     stream=None) -> Sparse24:
    rows, cols, ldw = _mat(W, name="W")
    out = Sparse24.empty(rows, cols, W.device) if out is None else out
    ldwm = 0
    if W_masked is not None:
        _, _, ldwm = _mat(W_masked, name="W_masked")
    d = out.c()
    _check(lib.prune24_compress(W.data_ptr(), rows, cols, ldw, C.byref(d), _ptr(W_masked), ldwm, _stream(stream)),
           "prune24_compress")
    return out


def prune24_transpose_repack(fwd: Sparse24, bwdT: Sparse24 | None = None, stream=None) -> Sparse24:
    bwdT = Sparse24.empty(fwd.cols, fwd.rows, fwd.vals.device) if bwdT is None else bwdT
    a, b = fwd.c(), bwdT.c()
    _check(lib.prune24_transpose_repack(C.byref(a), C.byref(b), _stream(stream)), "prune24_transpose_repack")
    return bwdT


def vnm24_compress(A: torch.Tensor, V: int, M: int, out: Sparse24 | None = None,
                   colidx: torch.Tensor | None = None, A_masked: torch.Tensor | None = None,
                   stream=None) -> tuple[torch.Tensor, Sparse24]:
    """V:2:M prune of A along its columns: (colidx uint8 [ceil(rows/V), cols/M, 4],
    the condensed [rows, 4 cols/M] matrix compressed 2:4). A_masked (optional, may be
    A itself) receives A with the pruned entries set to +0."""
    rows, cols, lda = _mat(A, name="A")
    if M <= 0 or cols % M:
        raise P24Error(P24_EINVAL, f"vnm24_compress: cols={cols} is not a multiple of M={M}")
    nb = (rows + V - 1) // V if V > 0 else 0
    out = Sparse24.empty(rows, 4 * (cols // M), A.device) if out is None else out
    if colidx is None:
        colidx = torch.empty((nb, cols // M, 4), dtype=torch.uint8, device=A.device)
    ldam = 0
    if A_masked is not None:
        _, _, ldam = _mat(A_masked, name="A_masked")
    d = out.c()
    _check(lib.vnm24_compress(A.data_ptr(), rows, cols, lda, V, M, colidx.data_ptr(), C.byref(d), _ptr(A_masked),
                              ldam, _stream(stream)), "vnm24_compress")
    return colidx, out


def vnm24_spmm(colidx: torch.Tensor, A: Sparse24, V: int, M: int, B: torch.Tensor, bias: torch.Tensor | None = None,
               relu: bool = False, Y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y = act(A . B + bias): A V:2:M-sparse (vnm24_compress's colidx and condensed
    matrix, pruned with V and M), B dense [K, N] with K = A.cols * M / 4."""
    K, N, ldb = _mat(B, name="B")
    if K != A.cols // 4 * M:
        raise ValueError(f"B has {K} rows; the V:2:M operand needs {A.cols // 4 * M}")
    Y = torch.empty((A.rows, N), dtype=torch.bfloat16, device=B.device) if Y is None else Y
    _, _, ldy = _mat(Y, name="Y")
    flags = (P24_EPI_BIAS if bias is not None else 0) | (P24_EPI_RELU if relu else 0)
    a = A.c()
    _check(lib.vnm24_spmm(colidx.data_ptr(), C.byref(a), V, M, B.data_ptr(), N, ldb, _ptr(bias), flags,
                          Y.data_ptr(), ldy, _stream(stream)), "vnm24_spmm")
    return Y


def prune24_compress_both(W: torch.Tensor, fwd: Sparse24 | None = None, bwdT: Sparse24 | None = None,
                          W_masked: torch.Tensor | None = None, stream=None) -> tuple[Sparse24, Sparse24]:
    rows, cols, ldw = _mat(W, name="W")
    fwd = Sparse24.empty(rows, cols, W.device) if fwd is None else fwd
    bwdT = Sparse24.empty(cols, rows, W.device) if bwdT is None else bwdT
    ldwm = 0
    if W_masked is not None:
        _, _, ldwm = _mat(W_masked, name="W_masked")
    a, b = fwd.c(), bwdT.c()
    _check(lib.prune24_compress_both(W.data_ptr(), rows, cols, ldw, C.byref(a), C.byref(b), _ptr(W_masked), ldwm,
                                     _stream(stream)), "prune24_compress_both")
    return fwd, bwdT


def spmm24_fwd(X: torch.Tensor, W: Sparse24, bias: torch.Tensor | None = None, relu: bool = False,
               act24: bool = False, Y: torch.Tensor | None = None, Y24: Sparse24 | None = None, stream=None,
               test_stall: bool = False):
    """Y = act(X W^T + bias); with act24 also returns the 2:4-compressed Y (Y, Y24).
    test_stall (test only): make the kernel's bounded waits expire (P24_EPI_TEST_STALL)."""
    M, K, ldx = _mat(X, name="X")
    N = W.rows
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device) if Y is None else Y
    _, _, ldy = _mat(Y, name="Y")
    flags = (P24_EPI_BIAS if bias is not None else 0) | (P24_EPI_RELU if relu else 0)
    if test_stall:
        flags |= P24_EPI_TEST_STALL
    y24c = None
    if act24:
        flags |= P24_EPI_ACT24
        Y24 = Sparse24.empty(M, N, X.device) if Y24 is None else Y24
        y24c = Y24.c()
    if bias is not None and (bias.dtype != torch.float32 or not bias.is_cuda):
        raise TypeError("bias must be a CUDA float32 tensor")
    w = W.c()
    _check(lib.spmm24_fwd(X.data_ptr(), M, ldx, C.byref(w), _ptr(bias), flags, Y.data_ptr(), ldy,
                          C.byref(y24c) if y24c is not None else None, _stream(stream)), "spmm24_fwd")
    return (Y, Y24) if act24 else Y


def spmm24_fwd_sparse_act(Xs: Sparse24, Wm: torch.Tensor, bias: torch.Tensor | None = None, relu: bool = False,
                          Y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    N, K, ldw = _mat(Wm, name="Wm")
    Y = torch.empty((Xs.rows, N), dtype=torch.bfloat16, device=Wm.device) if Y is None else Y
    _, _, ldy = _mat(Y, name="Y")
    flags = (P24_EPI_BIAS if bias is not None else 0) | (P24_EPI_RELU if relu else 0)
    x = Xs.c()
    _check(lib.spmm24_fwd_sparse_act(C.byref(x), Wm.data_ptr(), N, ldw, _ptr(bias), flags, Y.data_ptr(), ldy,
                                     _stream(stream)), "spmm24_fwd_sparse_act")
    return Y


def spmm24_bwd_dx(dY: torch.Tensor, WbwdT: Sparse24, gate: torch.Tensor | None = None,
                  dX: torch.Tensor | None = None, dbias: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """dX = (dY W_bwd) * [gate > 0]; with dbias (fp32 [K]) also its column sums, fused."""
    M, N, lddy = _mat(dY, name="dY")
    K = WbwdT.rows
    dX = torch.empty((M, K), dtype=torch.bfloat16, device=dY.device) if dX is None else dX
    _, _, lddx = _mat(dX, name="dX")
    ldg = 0
    if gate is not None:
        _, _, ldg = _mat(gate, name="gate")
    w = WbwdT.c()
    if dbias is not None and (dbias.dtype != torch.float32 or dbias.numel() != K or not dbias.is_contiguous()):
        raise ValueError(f"dbias must be a contiguous fp32 tensor of {K} elements")
    _check(lib.spmm24_bwd_dx(dY.data_ptr(), M, lddy, C.byref(w), _ptr(gate), ldg, dX.data_ptr(), lddx,
                             _ptr(dbias), _stream(stream)), "spmm24_bwd_dx")
    return dX


def spmm24_fwd_lowrank(X: torch.Tensor, W: Sparse24, T: torch.Tensor, L: torch.Tensor,
                       bias: torch.Tensor | None = None, relu: bool = False, Y: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """Y = act(X W^T + T L^T + bias): the sparse linear with SLOPE's low-rank adapter,
    T = X R^T [M, r] (see p24_gemm_nt), L [N, r]."""
    M, K, ldx = _mat(X, name="X")
    N = W.rows
    _, r, ldt = _mat(T, name="T")
    _, _, ldl = _mat(L, name="L")
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device) if Y is None else Y
    _, _, ldy = _mat(Y, name="Y")
    flags = (P24_EPI_BIAS if bias is not None else 0) | (P24_EPI_RELU if relu else 0)
    w = W.c()
    _check(lib.spmm24_fwd_lowrank(X.data_ptr(), M, ldx, C.byref(w), T.data_ptr(), ldt, L.data_ptr(), ldl, r,
                                  _ptr(bias), flags, Y.data_ptr(), ldy, None, _stream(stream)), "spmm24_fwd_lowrank")
    return Y


def spmm24_bwd_dx_lowrank(dY: torch.Tensor, WbwdT: Sparse24, U: torch.Tensor, Rt: torch.Tensor,
                          gate: torch.Tensor | None = None, dX: torch.Tensor | None = None,
                          dbias: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """dX = (dY W_bwd + U R) * [gate > 0]: U = dY L [M, r], Rt = R^T [K, r]."""
    M, N, lddy = _mat(dY, name="dY")
    K = WbwdT.rows
    _, r, ldu = _mat(U, name="U")
    _, _, ldrt = _mat(Rt, name="Rt")
    dX = torch.empty((M, K), dtype=torch.bfloat16, device=dY.device) if dX is None else dX
    _, _, lddx = _mat(dX, name="dX")
    ldg = 0 if gate is None else _mat(gate, name="gate")[2]
    w = WbwdT.c()
    _check(lib.spmm24_bwd_dx_lowrank(dY.data_ptr(), M, lddy, C.byref(w), U.data_ptr(), ldu, Rt.data_ptr(), ldrt, r,
                                     _ptr(gate), ldg, dX.data_ptr(), lddx, _ptr(dbias), _stream(stream)),
           "spmm24_bwd_dx_lowrank")
    return dX


def p24_gemm_nt(A: torch.Tensor, B: torch.Tensor, C_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """C = A B^T (bf16, fp32 accumulation): A [M, K], B [N, K]."""
    M, K, lda = _mat(A, name="A")
    N, K2, ldb = _mat(B, name="B")
    if K2 != K:
        raise ValueError("A and B need the same number of columns")
    Cm = torch.empty((M, N), dtype=torch.bfloat16, device=A.device) if C_out is None else C_out
    _, _, ldc = _mat(Cm, name="C")
    _check(lib.p24_gemm_nt(A.data_ptr(), M, lda, B.data_ptr(), N, ldb, K, Cm.data_ptr(), ldc, _stream(stream)),
           "p24_gemm_nt")
    return Cm


def p24_gemm_tn(A: torch.Tensor, B: torch.Tensor, C_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """C = A^T B (contraction over the rows M): A [M, N], B [M, K] -> C [N, K]."""
    M, N, lda = _mat(A, name="A")
    M2, K, ldb = _mat(B, name="B")
    if M2 != M:
        raise ValueError("A and B need the same number of rows")
    Cm = torch.empty((N, K), dtype=torch.bfloat16, device=A.device) if C_out is None else C_out
    _, _, ldc = _mat(Cm, name="C")
    _check(lib.p24_gemm_tn(A.data_ptr(), lda, B.data_ptr(), ldb, M, N, K, Cm.data_ptr(), ldc, _stream(stream)),
           "p24_gemm_tn")
    return Cm


def p24_transpose(src: torch.Tensor, dst: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    rows, cols, lds = _mat(src, name="src")
    dst = torch.empty((cols, rows), dtype=torch.bfloat16, device=src.device) if dst is None else dst
    _, _, ldd = _mat(dst, name="dst")
    _check(lib.p24_transpose(src.data_ptr(), rows, cols, lds, dst.data_ptr(), ldd, _stream(stream)), "p24_transpose")
    return dst


def masked_dw_gemm(dY: torch.Tensor, X: torch.Tensor, Wfwd: Sparse24, dW: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    M, N, lddy = _mat(dY, name="dY")
    M2, K, ldx = _mat(X, name="X")
    if M2 != M:
        raise ValueError("dY and X must have the same number of rows")
    dW = torch.empty((Wfwd.rows, Wfwd.cols), dtype=torch.bfloat16, device=dY.device) if dW is None else dW
    _, _, lddw = _mat(dW, name="dW")
    w = Wfwd.c()
    _check(lib.masked_dw_gemm(dY.data_ptr(), lddy, X.data_ptr(), ldx, M, C.byref(w), dW.data_ptr(), lddw,
                              _stream(stream)), "masked_dw_gemm")
    return dW


def p24_colsum(G: torch.Tensor, out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    M, N, ldg = _mat(G, name="G")
    out = torch.empty(N, dtype=torch.float32, device=G.device) if out is None else out
    need = int(lib.p24_colsum_workspace_size(M, N))
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=G.device)
    _check(lib.p24_colsum(G.data_ptr(), M, N, ldg, out.data_ptr(), ws.data_ptr(), ws.numel() * ws.element_size(),
                          _stream(stream)), "p24_colsum")
    return out


def p24_colsum_noalloc(G: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Column sums with the library's fixed device scratch (no workspace; see include/prune24.h)."""
    M, N, ldg = _mat(G, name="G")
    out = torch.empty(N, dtype=torch.float32, device=G.device) if out is None else out
    _check(lib.p24_colsum_noalloc(G.data_ptr(), M, N, ldg, out.data_ptr(), _stream(stream)), "p24_colsum_noalloc")
    return out


def ffn24_workspace_size_lowrank(M: int, d: int, ffn: int, act24: bool, r: int) -> int:
    return int(lib.ffn24_workspace_size_lowrank(M, d, ffn, (P24_STEP_ACT24 if act24 else 0) | P24_STEP_ADAPTERS, r))


def ffn24_workspace_size(M: int, d: int, ffn: int, act24: bool = False, vnm: tuple | None = None) -> int:
    if vnm:
        a = p24_ffn_args(M=M, d=d, ffn=ffn, flags=P24_STEP_VNM | (P24_STEP_ACT24 if act24 else 0),
                         vnm_V=int(vnm[0]), vnm_M=int(vnm[1]))
        return int(lib.ffn24_workspace_size_args(C.byref(a)))
    return int(lib.ffn24_workspace_size(M, d, ffn, P24_STEP_ACT24 if act24 else 0))


STEP_PHASES = 9
STEP_PHASE_NAMES = ("prune_up", "prune_down", "up_fwd", "down_fwd", "down_bwd_dx", "db_down", "dW_down",
                    "up_bwd_dx", "dW_up")


STEP_WEIGHTS = ("up_fwd", "up_bwdT", "down_fwd", "down_bwdT")


def ffn24_step(X, W_up, b_up, W_down, b_down, dY, act24: bool = False, out: dict | None = None,
               workspace: torch.Tensor | None = None, stream=None, events=None, weights: dict | None = None,
               keep_masks: bool = False, adapters: dict | None = None, vnm: tuple | None = None) -> dict:
    """One 2:4 FFN layer fwd+bwd; returns dict(Y, H, dX, dW_up, dW_down, db_up, db_down).

    events: optional ctypes array of 2 * STEP_PHASES raw cudaEvent_t handles, recorded
    before/after each phase (see ffn24_step_traced in include/prune24.h).
    weights: optional caller-owned compressed weights, a dict with Sparse24 entries
    up_fwd [ffn, d], up_bwdT [d, ffn], down_fwd [d, ffn], down_bwdT [ffn, d] and a bf16
    W_down_masked [d, ffn]. Without keep_masks the step prunes W_up / W_down afresh and
    writes the results there; with keep_masks=True it uses them as they are (fixed
    masks) and W_up / W_down are not read (they may be None).
    adapters: optional SLOPE low-rank adapters, a dict of bf16 tensors L_up [ffn, r],
    R_up [r, d], L_down [d, r], R_down [r, ffn]; their gradients come back as
    dL_up, dR_up, dL_down, dR_down (see include/prune24.h).
    A bf16 [M, ffn] tensor under out["dH"] receives the gated hidden gradient dH.
    vnm: (V, M) for V:N:M activations (P24_STEP_VNM): H is pruned V:2:M along ffn and
    the down forward runs as vnm24_spmm; the returned H is the pruned one."""
    M, d, _ = _mat(X, name="X")
    w = dict(weights or {})
    if keep_masks:
        missing = [k for k in STEP_WEIGHTS + (("W_down_masked",) if act24 else ()) if w.get(k) is None]
        if missing:
            raise ValueError(f"keep_masks needs the compressed weights: missing {missing}")
        ffn = w["up_fwd"].rows
    else:
        ffn = W_up.shape[0]
    dev = X.device
    for t, name, shape in ((W_up, "W_up", (ffn, d)), (W_down, "W_down", (d, ffn)), (dY, "dY", (M, d)),
                           (w.get("W_down_masked"), "W_down_masked", (d, ffn))):
        if t is None:
            continue
        _mat(t, name=name)
        if tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {shape} tensor")
    o = {} if out is None else dict(out)
    bf = torch.bfloat16
    o.setdefault("Y", torch.empty((M, d), dtype=bf, device=dev))
    o.setdefault("H", torch.empty((M, ffn), dtype=bf, device=dev))
    o.setdefault("dX", torch.empty((M, d), dtype=bf, device=dev))
    o.setdefault("dW_up", torch.empty((ffn, d), dtype=bf, device=dev))
    o.setdefault("dW_down", torch.empty((d, ffn), dtype=bf, device=dev))
    o.setdefault("db_up", torch.empty(ffn, dtype=torch.float32, device=dev))
    o.setdefault("db_down", torch.empty(d, dtype=torch.float32, device=dev))
    r = 0
    if adapters is not None:
        r = adapters["L_up"].shape[1]
        for k, shape in (("L_up", (ffn, r)), ("R_up", (r, d)), ("L_down", (d, r)), ("R_down", (r, ffn))):
            t = adapters[k]
            if t.dtype != bf or tuple(t.shape) != shape or not t.is_contiguous():
                raise ValueError(f"adapter {k} must be a contiguous bf16 {shape} tensor")
            o.setdefault("d" + k, torch.empty(shape, dtype=bf, device=dev))
    flags = ((P24_STEP_ACT24 if act24 else 0) | (P24_STEP_KEEP_MASKS if keep_masks else 0) |
             (P24_STEP_ADAPTERS if r else 0) | (P24_STEP_VNM if vnm else 0))
    a = p24_ffn_args(M, d, ffn, flags, X.data_ptr(), _ptr(W_up), _ptr(b_up),
                     _ptr(W_down), _ptr(b_down), dY.data_ptr(), o["Y"].data_ptr(), o["H"].data_ptr(),
                     o["dX"].data_ptr(), o["dW_up"].data_ptr(), o["dW_down"].data_ptr(), _ptr(o["db_up"]),
                     _ptr(o["db_down"]))
    a.r = r
    if vnm:
        a.vnm_V, a.vnm_M = int(vnm[0]), int(vnm[1])
    if workspace is None:
        workspace = torch.empty(int(lib.ffn24_workspace_size_args(C.byref(a))), dtype=torch.uint8, device=dev)
    structs = {k: w[k].c() for k in STEP_WEIGHTS if w.get(k) is not None}  # alive for the call
    for k, st in structs.items():
        setattr(a, k, C.pointer(st))
    a.W_down_masked = _ptr(w.get("W_down_masked"))
    if o.get("dH") is not None:
        _mat(o["dH"], name="dH")
        if tuple(o["dH"].shape) != (M, ffn) or not o["dH"].is_contiguous():
            raise ValueError(f"dH must be a contiguous {(M, ffn)} tensor")
        a.dH = o["dH"].data_ptr()
    if r:
        for k in ("L_up", "R_up", "L_down", "R_down"):
            setattr(a, k, adapters[k].data_ptr())
            setattr(a, "d" + k, o["d" + k].data_ptr())
    if events is None:
        _check(lib.ffn24_step(C.byref(a), workspace.data_ptr(), workspace.numel(), _stream(stream)), "ffn24_step")
    else:
        _check(lib.ffn24_step_traced(C.byref(a), workspace.data_ptr(), workspace.numel(), _stream(stream),
                                     C.cast(events, C.POINTER(C.c_void_p)), len(events)), "ffn24_step_traced")
    return o


def p24_launch_count() -> int:
    return int(lib.p24_launch_count())


def p24_selftest_timeout(limit_ns: int = 10_000_000, stream=None) -> None:
    """Launch the bounded-wait failure self test (see include/prune24.h)."""
    _check(lib.p24_selftest_timeout(limit_ns, _stream(stream)), "p24_selftest_timeout")


def p24_query_timeout(stream=None) -> tuple[int, int, int]:
    """(status, CTA, barrier shared address) of the first expired wait since the last
    query (-1, -1 when none); clears the status."""
    cta, bar = C.c_int64(-1), C.c_int64(-1)
    code = int(lib.p24_query_timeout(_stream(stream), C.byref(cta), C.byref(bar)))
    return code, cta.value, bar.value


def p24_query_status(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device status word."""
    return int(lib.p24_query_status(_stream(stream)))


@dataclass
class Hybrid:
    """Hybrid ELL + dense-overflow form of a [rows, cols] bf16 matrix (see p24_hybrid in
    include/prune24.h): device tensors nnz, ell_cols, ell_vals, slot, ovf_rows, n_ovf, ovf."""
    nnz: torch.Tensor
    ell_cols: torch.Tensor
    ell_vals: torch.Tensor
    slot: torch.Tensor
    ovf_rows: torch.Tensor
    n_ovf: torch.Tensor
    ovf: torch.Tensor
    rows: int
    cols: int
    E: int
    cap: int

    @staticmethod
    def empty(rows: int, cols: int, E: int, cap: int, device="cuda") -> "Hybrid":
        i32 = torch.int32
        return Hybrid(torch.empty(rows, dtype=i32, device=device),
                      torch.empty((rows, E), dtype=torch.int16, device=device),   # uint16 column bits
                      torch.empty((rows, E), dtype=torch.bfloat16, device=device),
                      torch.empty(rows, dtype=i32, device=device), torch.empty(max(cap, 1), dtype=i32, device=device),
                      torch.empty(1, dtype=i32, device=device),
                      torch.empty((max(cap, 1), cols), dtype=torch.bfloat16, device=device), rows, cols, E, cap)

    def c(self) -> p24_hybrid:
        return p24_hybrid(self.rows, self.cols, self.E, self.cap, self.nnz.data_ptr(), self.ell_cols.data_ptr(),
                          self.ell_vals.data_ptr(), self.slot.data_ptr(), self.ovf_rows.data_ptr(),
                          self.n_ovf.data_ptr(), self.ovf.data_ptr(), self.ovf.stride(0))


def hyb_compress(A: torch.Tensor, E: int, cap: int, out: Hybrid | None = None, stream=None) -> Hybrid:
    """The hybrid form of A (ELL width E, backup capacity cap)."""
    rows, cols, lda = _mat(A, name="A")
    out = Hybrid.empty(rows, cols, E, cap, A.device) if out is None else out
    h = out.c()
    _check(lib.hyb_compress(A.data_ptr(), lda, C.byref(h), _stream(stream)), "hyb_compress")
    return out


def hyb_spmm(h: Hybrid, B: torch.Tensor, Y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Hybrid to dense: Y = A . B, B [cols, N]."""
    K, N, ldb = _mat(B, name="B")
    Y = torch.empty((h.rows, N), dtype=torch.bfloat16, device=B.device) if Y is None else Y
    _, _, ldy = _mat(Y, name="Y")
    hc = h.c()
    _check(lib.hyb_spmm(C.byref(hc), B.data_ptr(), N, ldb, Y.data_ptr(), ldy, _stream(stream)), "hyb_spmm")
    return Y


def hyb_sddmm(h: Hybrid, G: torch.Tensor, B: torch.Tensor, S_ell: torch.Tensor | None = None,
              S_ovf: torch.Tensor | None = None, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Dense to hybrid: (G . B^T) at A's nonzeros, in A's layout: (S_ell [rows, E], S_ovf [cap, cols])."""
    R, N, ldg = _mat(G, name="G")
    _, _, ldb = _mat(B, name="B")
    S_ell = torch.empty((h.rows, h.E), dtype=torch.bfloat16, device=G.device) if S_ell is None else S_ell
    S_ovf = torch.empty((max(h.cap, 1), h.cols), dtype=torch.bfloat16, device=G.device) if S_ovf is None else S_ovf
    hc = h.c()
    _check(lib.hyb_sddmm(C.byref(hc), G.data_ptr(), N, ldg, B.data_ptr(), ldb, S_ell.data_ptr(), S_ovf.data_ptr(),
                         S_ovf.stride(0), _stream(stream)), "hyb_sddmm")
    return S_ell, S_ovf
