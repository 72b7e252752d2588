"""C-ABI checks that need no GPU: the library loads, exports every function
include/prune24.h declares, computes its stride helpers, and rejects bad
arguments on the host before touching CUDA."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def native():
    from semi_structured_sparse_prune24_gb300 import _native
    return _native


def declared_functions():
    src = open(os.path.join(ROOT, "include", "prune24.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\*?\s*([A-Za-z_]\w*)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("prune24_compress", "prune24_transpose_repack", "spmm24_fwd", "spmm24_bwd_dx",
                     "masked_dw_gemm", "ffn24_step"):
        assert required in names


def test_every_declared_function_is_exported(native):
    lib = C.CDLL(native._LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_stride_helpers(native):
    L = native.lib
    assert L.p24_ld_vals(8200) == 4104 and L.p24_ld_meta(8200) == 1040
    assert L.p24_ld_vals(512) == 256 and L.p24_ld_meta(512) == 64
    assert L.p24_ld_vals(4) == 8 and L.p24_ld_meta(4) == 16
    for cols in range(4, 2000, 4):
        assert L.p24_ld_vals(cols) >= cols // 2 and L.p24_ld_vals(cols) % 8 == 0
        assert L.p24_ld_meta(cols) * 2 >= cols // 4 and L.p24_ld_meta(cols) % 16 == 0


def test_strerror(native):
    for code in range(-6, 1):
        assert native.lib.p24_strerror(code)
    assert b"unknown" in native.lib.p24_strerror(-99)


def _sp(vals, meta, rows, cols, ldv, ldm, native):
    return native.p24_sparse(vals, meta, rows, cols, ldv, ldm)


def test_host_validation_rejects_before_launch(native):
    L = native.lib
    EINVAL, EALIGN = native.P24_EINVAL, native.P24_EALIGN
    fake = 0x10000  # never dereferenced: every call below fails validation first
    good = _sp(fake, fake, 8, 16, 8, 16, native)
    # null input
    assert L.prune24_compress(None, 8, 16, 16, C.byref(good), None, 0, None) == EINVAL
    # cols not a multiple of 4
    assert L.prune24_compress(fake, 8, 18, 24, C.byref(good), None, 0, None) == EINVAL
    # misaligned input pointer / stride
    assert L.prune24_compress(fake + 2, 8, 16, 16, C.byref(good), None, 0, None) == EALIGN
    assert L.prune24_compress(fake, 8, 16, 20, C.byref(good), None, 0, None) == EALIGN
    # output descriptor with a too-small metadata stride
    bad = _sp(fake, fake, 8, 16, 8, 8, native)
    assert L.prune24_compress(fake, 8, 16, 16, C.byref(bad), None, 0, None) == EINVAL
    # shape mismatch between input and descriptor
    assert L.prune24_compress(fake, 4, 16, 16, C.byref(good), None, 0, None) == EINVAL
    # repack needs rows % 4 == 0 and transposed shapes
    odd = _sp(fake, fake, 6, 16, 8, 16, native)
    t = _sp(fake, fake, 16, 6, 8, 16, native)
    assert L.prune24_transpose_repack(C.byref(odd), C.byref(t), None) == EINVAL
    # GEMMs: bad flags, missing bias, K % 8
    w = _sp(fake, fake, 16, 16, 8, 16, native)
    assert L.spmm24_fwd(fake, 8, 16, C.byref(w), None, 0x80, fake, 16, None, None) == EINVAL
    assert L.spmm24_fwd(fake, 8, 16, C.byref(w), None, native.P24_EPI_BIAS, fake, 16, None, None) == EINVAL
    w12 = _sp(fake, fake, 16, 12, 8, 16, native)
    assert L.spmm24_fwd(fake, 8, 16, C.byref(w12), None, 0, fake, 16, None, None) == EINVAL
    assert L.spmm24_bwd_dx(None, 8, 16, C.byref(w), None, 0, fake, 16, None, None) == EINVAL
    # fused bias gradient must be 16-byte aligned
    assert L.spmm24_bwd_dx(fake, 8, 16, C.byref(w), None, 0, fake, 16, fake + 4, None) == native.P24_EALIGN
    assert L.masked_dw_gemm(fake, 16, fake, 16, 8, None, fake, 16, None) == EINVAL
    # colsum workspace too small
    assert L.p24_colsum(fake, 100, 16, 16, fake, fake, 8, None) == native.P24_ENOSPACE
    # ffn step: null args, bad flags, d % 8
    assert L.ffn24_step(None, fake, 1 << 20, None) == EINVAL
    a = native.p24_ffn_args(8, 12, 16, 0, fake, fake, None, fake, None, fake, fake, fake, fake, fake, fake,
                            None, None)
    assert L.ffn24_step(C.byref(a), fake, 1 << 30, None) == EINVAL
    a.d, a.flags = 16, 0x8
    assert L.ffn24_step(C.byref(a), fake, 1 << 30, None) == EINVAL
    # fixed masks need the caller's compressed weights (and W_down on its mask with ACT24)
    a.flags = native.P24_STEP_KEEP_MASKS
    assert L.ffn24_step(C.byref(a), fake, 1 << 30, None) == EINVAL
    up, upT = _sp(fake, fake, 16, 16, 8, 16, native), _sp(fake, fake, 16, 16, 8, 16, native)
    dn, dnT = _sp(fake, fake, 16, 16, 8, 16, native), _sp(fake, fake, 16, 16, 8, 16, native)
    a.up_fwd, a.up_bwdT, a.down_fwd, a.down_bwdT = (C.pointer(x) for x in (up, upT, dn, dnT))
    a.flags = native.P24_STEP_KEEP_MASKS | native.P24_STEP_ACT24
    assert L.ffn24_step(C.byref(a), fake, 1 << 30, None) == EINVAL
    # a compressed weight of the wrong shape
    a.flags = native.P24_STEP_KEEP_MASKS
    a.up_fwd = C.pointer(_sp(fake, fake, 16, 8, 8, 16, native))
    assert L.ffn24_step(C.byref(a), fake, 1 << 30, None) == EINVAL


def test_workspace_sizes_grow_with_the_problem(native):
    f = native.lib.ffn24_workspace_size
    assert f(128, 256, 512, 0) < f(256, 256, 512, 0) < f(256, 256, 512, native.P24_STEP_ACT24)
    assert native.lib.p24_colsum_workspace_size(64, 100) == 400
    assert native.lib.p24_colsum_workspace_size(10 ** 6, 8) == 1024 * 8 * 4


def test_host_validation_of_the_fused_lowrank_dense_and_colsum_calls(native):
    L = native.lib
    EINVAL, EALIGN, ENOSPACE = native.P24_EINVAL, native.P24_EALIGN, native.P24_ENOSPACE
    fake = 0x10000  # never dereferenced: every call below fails validation first
    fwd = _sp(fake, fake, 16, 32, 16, 16, native)      # W [16, 32]
    bwdT = _sp(fake, fake, 32, 16, 8, 16, native)      # W_bwd^T [32, 16]
    # fused prune-both: rows and cols multiples of 4, transposed descriptor shapes, aligned masked copy
    assert L.prune24_compress_both(fake, 14, 32, 32, C.byref(fwd), C.byref(bwdT), None, 0, None) == EINVAL
    assert L.prune24_compress_both(fake, 16, 30, 32, C.byref(fwd), C.byref(bwdT), None, 0, None) == EINVAL
    same = _sp(fake, fake, 16, 32, 16, 16, native)
    assert L.prune24_compress_both(fake, 16, 32, 32, C.byref(fwd), C.byref(same), None, 0, None) == EINVAL
    assert L.prune24_compress_both(fake, 16, 32, 32, C.byref(fwd), C.byref(bwdT), fake + 2, 32, None) == EALIGN
    # allocation-free colsum: wider than its fixed scratch
    wide = (1 << 20) + 8
    assert L.p24_colsum_noalloc(fake, 4, wide, wide, fake, None) == ENOSPACE
    # low-rank calls: rank a multiple of 8, 16-byte factor strides, factors present
    w = _sp(fake, fake, 16, 16, 8, 16, native)
    assert L.spmm24_fwd_lowrank(fake, 8, 16, C.byref(w), fake, 12, fake, 12, 12, None, 0, fake, 16, None,
                                None) == EINVAL
    assert L.spmm24_fwd_lowrank(fake, 8, 16, C.byref(w), fake, 20, fake, 16, 16, None, 0, fake, 16, None,
                                None) == EALIGN
    assert L.spmm24_bwd_dx_lowrank(fake, 8, 16, C.byref(w), fake, 16, None, 16, 16, None, 0, fake, 16, None,
                                   None) == EINVAL
    # dense rank-r products: K >= 0, strides cover the rows and are multiples of 8 elements
    assert L.p24_gemm_nt(fake, 8, 16, fake, 8, 16, -1, fake, 8, None) == EINVAL
    assert L.p24_gemm_nt(fake, 8, 8, fake, 8, 16, 16, fake, 8, None) == EINVAL
    assert L.p24_gemm_tn(fake, 16, fake, 20, 8, 16, 16, fake, 16, None) == EALIGN
    # transpose: 2-byte alignment, strides cover the rows
    assert L.p24_transpose(fake + 1, 4, 4, 4, fake, 4, None) == EALIGN
    assert L.p24_transpose(fake, 4, 8, 4, fake, 4, None) == EINVAL


def test_host_validation_of_vnm24_compress(native):
    L = native.lib
    EINVAL, EALIGN = native.P24_EINVAL, native.P24_EALIGN
    fake = 0x10000  # never dereferenced: every call below fails validation first
    out = _sp(fake, fake, 8, 16, 8, 16, native)          # condensed [8, 4*32/8 = 16]
    assert L.vnm24_compress(fake, 8, 32, 32, 4, 12, fake, C.byref(out), None, 0, None) == EINVAL   # M not dividing 256
    assert L.vnm24_compress(fake, 8, 32, 32, 4, 256, fake, C.byref(out), None, 0, None) == EINVAL  # M above 128
    assert L.vnm24_compress(fake, 8, 36, 40, 4, 8, fake, C.byref(out), None, 0, None) == EINVAL    # cols % M
    assert L.vnm24_compress(fake, 8, 32, 32, 0, 8, fake, C.byref(out), None, 0, None) == EINVAL    # V < 1
    assert L.vnm24_compress(fake, 8, 32, 36, 4, 8, fake, C.byref(out), None, 0, None) == EALIGN    # lda % 8
    assert L.vnm24_compress(fake, 8, 32, 32, 4, 16, fake, C.byref(out), None, 0, None) == EINVAL   # out is not [8, 8]
    assert L.vnm24_compress(fake, 8, 32, 32, 4, 8, None, C.byref(out), None, 0, None) == EINVAL    # no colidx


def test_host_validation_of_vnm24_compress_masked_and_spmm(native):
    L = native.lib
    EINVAL, EALIGN, EUNS = native.P24_EINVAL, native.P24_EALIGN, native.P24_EUNSUPPORTED
    fake = 0x10000  # never dereferenced: every call below fails validation first
    out = _sp(fake, fake, 8, 16, 8, 16, native)
    # masked output: in place needs the same stride; V above 256 is not supported with it
    assert L.vnm24_compress(fake, 8, 32, 32, 4, 8, fake, C.byref(out), fake, 40, None) == EINVAL
    assert L.vnm24_compress(fake, 8, 32, 32, 300, 8, fake, C.byref(out), fake + 0x1000, 32, None) == EUNS
    assert L.vnm24_compress(fake, 8, 32, 32, 4, 8, fake, C.byref(out), fake + 8, 32, None) == EALIGN
    # vnm24_spmm: A condensed [512, 256] from K = 512 (M = 8); B [512, 256]
    a = _sp(fake, fake, 512, 256, 128, 32, native)
    assert L.vnm24_spmm(fake, C.byref(a), 256, 8, fake, 256, 256, None, 0x8, fake, 256, None) == EINVAL  # flag
    assert L.vnm24_spmm(fake, C.byref(a), 256, 12, fake, 256, 256, None, 0, fake, 256, None) == EINVAL   # M
    assert L.vnm24_spmm(fake, C.byref(a), 0, 8, fake, 256, 256, None, 0, fake, 256, None) == EINVAL      # V
    assert L.vnm24_spmm(fake, C.byref(a), 256, 8, fake, 256, 200, None, 0, fake, 256, None) == EINVAL    # ldb < N
    assert L.vnm24_spmm(fake, C.byref(a), 256, 8, fake, 256, 256, None, 1, fake, 256, None) == EINVAL    # bias
    assert L.vnm24_spmm(None, C.byref(a), 256, 8, fake, 256, 256, None, 0, fake, 256, None) == EINVAL    # colidx
    assert L.vnm24_spmm(fake + 4, C.byref(a), 256, 8, fake, 256, 256, None, 0, fake, 256, None) == EALIGN
    assert L.vnm24_spmm(fake, C.byref(a), 128, 8, fake, 256, 256, None, 0, fake, 256, None) == EUNS      # V % 256
    assert L.vnm24_spmm(fake, C.byref(a), 256, 8, fake, 264, 264, None, 0, fake, 264, None) == EUNS      # N % 256
    a2 = _sp(fake, fake, 512, 192, 96, 32, native)                                                      # 192 % 128
    assert L.vnm24_spmm(fake, C.byref(a2), 256, 8, fake, 256, 256, None, 0, fake, 256, None) == EUNS


def test_host_validation_of_the_hybrid_calls(native):
    L = native.lib
    EINVAL, EALIGN = native.P24_EINVAL, native.P24_EALIGN
    fake = 0x10000  # never dereferenced: every call below fails validation first
    H = native.p24_hybrid
    good = dict(rows=8, cols=64, E=4, cap=2, nnz=fake, ell_cols=fake, ell_vals=fake, slot=fake, ovf_rows=fake,
                n_ovf=fake, ovf=fake, ldo=64)
    def h(**kw):
        return H(**{**good, **kw})
    assert L.hyb_compress(fake, 64, C.byref(h(cols=60)), None) == EINVAL          # cols % 8
    assert L.hyb_compress(fake, 64, C.byref(h(cols=65544)), None) == EINVAL       # > 65536 columns
    assert L.hyb_compress(fake, 64, C.byref(h(E=0)), None) == EINVAL
    assert L.hyb_compress(fake, 64, C.byref(h(nnz=None)), None) == EINVAL
    assert L.hyb_compress(fake, 64, C.byref(h(slot=fake + 2)), None) == EALIGN
    assert L.hyb_compress(fake, 64, C.byref(h(ell_vals=fake + 4)), None) == EALIGN
    assert L.hyb_compress(fake, 60, C.byref(h()), None) == EINVAL                 # lda < cols
    assert L.hyb_spmm(C.byref(h()), fake, 12, 16, fake, 16, None) == EINVAL       # N % 8
    assert L.hyb_sddmm(C.byref(h()), fake, 40000, 40000, fake, 40000, fake, fake, 64, None) == EINVAL  # N cap
    assert L.hyb_sddmm(C.byref(h()), fake, 16, 16, fake, 16, fake + 2, fake, 64, None) == EALIGN
