"""The C ABI without a GPU: the library builds, loads, exports every symbol
include/rg.h declares, and rejects bad arguments on the host before any CUDA
call (no call here passes validation, so nothing is ever launched)."""
import ctypes
import os
import re

import pytest

from quantized_weight_out_gb300 import binding as rg
from quantized_weight_out_gb300 import build as rgbuild
from quantized_weight_out_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    rgbuild.build()
    return rg.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "rg.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(rg_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "rg_out_prod" in names and "rg_dequant" in names
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(n for n, _, _ in rg.SIGNATURES) == names


def test_noalloc_scratch_size_matches_the_header():
    """The binding's copy of RG_NOALLOC_SCRATCH_BYTES is the header's."""
    src = open(os.path.join(ROOT, "include", "rg.h")).read()
    m = re.search(r"#define\s+RG_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", src)
    assert m, "RG_NOALLOC_SCRATCH_BYTES not found in include/rg.h"
    assert rg.RG_NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_row_bytes_matches_block_sizes(lib):
    for wt in inputs.ALL_TYPES:
        for K in (0, 8, 32, 256, 4096, 14336, 17408, 300):
            assert rg.rg_row_bytes(wt, K) == inputs.row_bytes(wt, K), (wt, K)
    assert rg.rg_row_bytes(16, 256) == 0 and rg.rg_row_bytes(inputs.Q8_0, -32) == 0
    assert rg.rg_row_bytes(0, 256) == 0


def test_strerror_and_version(lib):
    for s in (0, -1, -2, -3, -4, -5, -6):
        assert rg.strerror(s) and rg.strerror(s) != "unknown status"
    assert rg.strerror(42) == "unknown status"
    assert rg.rg_version() >= 1


def test_dispatch(lib):
    assert rg.rg_select_variant(inputs.Q8_0, 4096, 4096, 2) == rg.RG_VARIANT_SMALLT
    assert rg.rg_select_variant(inputs.Q8_0, 256, 256, 32) == rg.RG_VARIANT_SMALLT   # 4 MFLOP
    assert rg.rg_select_variant(inputs.Q8_0, 4096, 4096, 32) == rg.RG_VARIANT_TC
    assert rg.rg_select_variant(inputs.Q4_K, 14336, 4096, 2048) == rg.RG_VARIANT_TC
    assert rg.rg_select_variant(inputs.Q4_K, 14336, 4096, 4) == rg.RG_VARIANT_SMALLT
    assert rg.rg_select_variant(inputs.Q4_K, 14336, 4096, 5) == rg.RG_VARIANT_TC
    assert rg.rg_select_variant(inputs.Q8_0, 14336, 4096, 4) == rg.RG_VARIANT_SMALLT
    assert rg.rg_select_variant(inputs.Q8_0, 14336, 4096, 5) == rg.RG_VARIANT_TC
    assert rg.rg_select_variant(inputs.Q4_0, 14336, 4096, 4) == rg.RG_VARIANT_TC
    # Q6_K rows are 16-byte aligned only for K % 2048 == 0; other K run on the SIMT variant
    assert rg.rg_select_variant(inputs.Q6_K, 4096, 4096, 2048) == rg.RG_VARIANT_TC
    assert rg.rg_select_variant(inputs.Q6_K, 4096, 5120, 2048) == rg.RG_VARIANT_SIMT32
    # Q3_K likewise; Q2_K rows (84 B per 256 values) need K % 1024 == 0
    assert rg.rg_select_variant(inputs.Q3_K, 4096, 4096, 2048) == rg.RG_VARIANT_TC
    assert rg.rg_select_variant(inputs.Q3_K, 4096, 5120, 2048) == rg.RG_VARIANT_SIMT32
    assert rg.rg_select_variant(inputs.Q2_K, 4096, 5120, 2048) == rg.RG_VARIANT_TC
    assert rg.rg_select_variant(inputs.Q2_K, 4096, 4864, 2048) == rg.RG_VARIANT_SIMT32
    # MXFP4 rows (136 B per 256 values) need K % 512 == 0
    assert rg.rg_select_variant(inputs.MXFP4, 4096, 4608, 2048) == rg.RG_VARIANT_TC
    assert rg.rg_select_variant(inputs.MXFP4, 4096, 4352, 2048) == rg.RG_VARIANT_SIMT32
    # (with a device the plan may add partial-sum slabs after the 16-bit copy of dY)
    assert rg.rg_workspace_bytes(rg.RG_VARIANT_TC, inputs.Q4_K, 14336, 4096, 2048) >= 2048 * 14336 * 2
    assert rg.rg_workspace_bytes(rg.RG_VARIANT_TC, inputs.Q4_K, 13, 4096, 3) == 3 * 16 * 2 + 160
    assert rg.rg_workspace_bytes(rg.RG_VARIANT_SIMT32, inputs.Q4_K, 14336, 4096, 8) == 0


def test_plan_validates_before_needing_a_device(lib):
    info = rg.rg_plan_info()
    assert rg.rg_plan(0, 16, 64, 256, 8, info) == rg.RG_ERR_TYPE
    assert rg.rg_plan(6, inputs.Q8_0, 64, 256, 8, info) == rg.RG_ERR_TYPE
    assert rg.rg_plan(0, inputs.Q8_0, 64, 200, 8, info) == rg.RG_ERR_SHAPE
    assert rg.rg_plan(0, inputs.F16, 64, 12, 8, info) == rg.RG_ERR_SHAPE
    assert rg.rg_plan(0, inputs.Q8_0, -1, 256, 8, info) == rg.RG_ERR_ARG
    assert rg.rg_plan(0, inputs.Q8_0, 64, 256, 1 << 31, info) == rg.RG_ERR_ARG
    assert lib.rg_plan(0, inputs.Q8_0, 64, 256, 8, None) == rg.RG_ERR_ARG
    assert ctypes.sizeof(rg.rg_plan_info) == 48
    assert rg.rg_launch_count() >= 0


BAD = 0x1000  # never dereferenced: every case below fails validation first


@pytest.mark.parametrize("args,status", [
    ((16, BAD, 64, 256, BAD, 8, BAD, 0.0), rg.RG_ERR_TYPE),
    ((0, BAD, 64, 256, BAD, 8, BAD, 0.0), rg.RG_ERR_TYPE),
    ((inputs.Q5_K, BAD, 64, 128, BAD, 8, BAD, 0.0), rg.RG_ERR_SHAPE),
    ((inputs.Q5_0, BAD, 64, 32, BAD, 8, BAD, 0.0), rg.RG_ERR_SHAPE),
    ((inputs.Q4_K, BAD, 64, 200, BAD, 8, BAD, 0.0), rg.RG_ERR_SHAPE),
    ((inputs.Q8_0, BAD, 64, 32, BAD, 8, BAD, 0.0), rg.RG_ERR_SHAPE),
    ((inputs.F16, BAD, 64, 12, BAD, 8, BAD, 0.0), rg.RG_ERR_SHAPE),
    ((inputs.Q4_0, BAD, -1, 256, BAD, 8, BAD, 0.0), rg.RG_ERR_ARG),
    ((inputs.Q4_0, BAD, 64, 256, BAD, 1 << 31, BAD, 0.0), rg.RG_ERR_ARG),
    ((inputs.Q4_0, None, 64, 256, BAD, 8, BAD, 0.0), rg.RG_ERR_ARG),
    ((inputs.Q4_0, BAD, 64, 256, None, 8, BAD, 0.0), rg.RG_ERR_ARG),
    ((inputs.Q4_0, BAD, 64, 256, BAD, 8, None, 0.0), rg.RG_ERR_ARG),
    ((inputs.Q4_0, BAD + 4, 64, 256, BAD, 8, BAD, 0.0), rg.RG_ERR_ALIGN),
    ((inputs.Q4_0, BAD, 64, 256, BAD + 8, 8, BAD, 0.0), rg.RG_ERR_ALIGN),
    ((inputs.Q4_0, BAD, 64, 256, BAD, 8, BAD + 2, 0.0), rg.RG_ERR_ALIGN),
    ((inputs.Q4_0, None, 64, 256, None, 0, None, 0.0), rg.RG_OK),     # T == 0: empty output
    ((inputs.Q4_0, None, 64, 0, None, 8, None, 0.0), rg.RG_OK),       # K == 0: empty output
])
def test_validation_before_any_launch(lib, args, status):
    assert rg.rg_out_prod(*args) == status
    assert rg.rg_out_prod_variant(rg.RG_VARIANT_SIMT32, *args) == status


def test_bad_variant_and_workspace(lib):
    # valid shapes but a bad variant id: rejected (the variant check follows
    # argument validation, and the empty case returns before it)
    assert rg.rg_out_prod_variant(7, 16, BAD, 64, 256, BAD, 8, BAD, 0.0) == rg.RG_ERR_TYPE


def test_dequant_validation(lib):
    assert rg.rg_dequant(16, BAD, 4, 256, BAD) == rg.RG_ERR_TYPE
    assert rg.rg_dequant(inputs.Q4_K, BAD, 4, 128, BAD) == rg.RG_ERR_SHAPE
    assert rg.rg_dequant(inputs.Q8_0, None, 4, 256, BAD) == rg.RG_ERR_ARG
    assert rg.rg_dequant(inputs.Q8_0, BAD + 1, 4, 256, BAD) == rg.RG_ERR_ALIGN
    assert rg.rg_dequant(inputs.Q8_0, None, 0, 256, None) == rg.RG_OK
    assert rg.rg_debug_wait_probe(0) == rg.RG_ERR_ARG


def test_product_path_has_no_cpu_fallback(lib, tmp_path):
    """The binding raises when the library is missing instead of computing."""
    saved = rg._lib
    rg._lib = None
    try:
        with pytest.raises(RuntimeError, match="no CPU fallback"):
            rg.load(str(tmp_path / "librg.so"))
    finally:
        rg._lib = saved
    src = open(os.path.join(ROOT, "quantized_weight_out_gb300", "binding.py")).read()
    assert "oracle" not in src and "numpy" not in src


def test_out_prod_ex_validation_before_any_launch(lib):
    """The strided / batched entry checks every batch on the host first."""
    A = 0x1000
    base = dict(variant=0, wtype=inputs.Q8_0, W=A, N=64, K=256, w_batch_bytes=0, dY=A, T=8,
                dy_t=64, dy_n=1, dy_batch=0, dX=A, dx_t=256, dx_batch=0, batch=2, beta=0.0)

    def call(**kw):
        a = dict(base, **kw)
        return rg.rg_out_prod_ex(a["variant"], a["wtype"], a["W"], a["N"], a["K"], a["w_batch_bytes"],
                                 a["dY"], a["T"], a["dy_t"], a["dy_n"], a["dy_batch"], a["dX"],
                                 a["dx_t"], a["dx_batch"], a["batch"], a["beta"])
    assert call(batch=0) == rg.RG_OK
    assert call(batch=-1) == rg.RG_ERR_ARG
    assert call(dx_t=255) == rg.RG_ERR_ARG              # rows shorter than K
    assert call(dx_t=258) == rg.RG_ERR_ALIGN            # dX rows not 16-byte aligned
    assert call(dy_n=0) == rg.RG_ERR_ARG
    assert call(w_batch_bytes=8) == rg.RG_ERR_ALIGN
    assert call(dx_batch=6) == rg.RG_ERR_ALIGN
    assert call(dY=A + 2, dy_t=1, dy_n=8) == rg.RG_ERR_ALIGN
    assert call(dY=A + 4) == rg.RG_ERR_ALIGN            # contiguous rows need 16-byte alignment
    assert call(wtype=16) == rg.RG_ERR_TYPE


def test_out_prod_batched_validation_before_any_launch(lib):
    """The two-dimension batched entry: weight counts must divide the
    gradient's batch counts, strides be non-negative and aligned, and every
    batch pass the row rules, all before any launch."""
    A = 0x1000
    base = dict(variant=0, wtype=inputs.Q8_0, W=A, N=64, K=256, w_n2=2, w_n3=1, w_s2=64 * 272,
                w_s3=0, dY=A, T=8, dy_t=64, dy_n=1, dy_s2=8 * 64, dy_s3=0, dX=A, dx_t=256,
                dx_s2=8 * 256, dx_s3=0, n2=4, n3=1, beta=0.0)

    def call(**kw):
        a = dict(base, **kw)
        return rg.rg_out_prod_batched(*[a[k] for k in base])
    assert call(n2=0) == rg.RG_OK and call(n3=0) == rg.RG_OK
    assert call(n2=-1) == rg.RG_ERR_ARG
    assert call(w_n2=0) == rg.RG_ERR_ARG
    assert call(w_n2=3) == rg.RG_ERR_SHAPE              # 3 weights for 4 batches
    assert call(n3=3, w_n3=2) == rg.RG_ERR_SHAPE
    assert call(w_s2=-16) == rg.RG_ERR_ARG
    assert call(w_s2=8) == rg.RG_ERR_ALIGN
    assert call(dx_s3=2, n3=2) == rg.RG_ERR_ALIGN
    assert call(dx_t=255) == rg.RG_ERR_ARG
    assert call(dY=A + 4) == rg.RG_ERR_ALIGN
    assert call(W=A + 8, w_n2=1) == rg.RG_ERR_ALIGN
    assert call(wtype=16) == rg.RG_ERR_TYPE


def test_mul_mat_validation(lib):
    A = 0x1000
    assert rg.rg_mul_mat(16, A, 64, 256, A, 4, A, 0.0) == rg.RG_ERR_TYPE
    assert rg.rg_mul_mat(inputs.Q8_0, A, 60, 256, A, 4, A, 0.0) == rg.RG_ERR_SHAPE
    assert rg.rg_mul_mat(inputs.Q8_0, A, 64, 255, A, 4, A, 0.0) == rg.RG_ERR_SHAPE
    assert rg.rg_mul_mat(inputs.Q8_0, A, 64, 256, A, 0, A, 0.0) == rg.RG_OK
    assert rg.rg_mul_mat(inputs.Q8_0, A + 4, 64, 256, A, 4, A, 0.0) == rg.RG_ERR_ALIGN
    assert rg.rg_mul_mat(inputs.Q8_0, A, 64, 256, A, 4, None, 0.0) == rg.RG_ERR_ARG
    # the forward's routes: auto, tensor core and small-T; no SIMT or forced tile shape
    for v in (rg.RG_VARIANT_SIMT32, rg.RG_VARIANT_TC_SINGLE, rg.RG_VARIANT_TC_PAIR, 9, -1):
        assert rg.rg_mul_mat_variant(v, inputs.Q8_0, A, 64, 256, A, 4, A, 0.0) == rg.RG_ERR_TYPE
    assert rg.rg_mul_mat_variant(rg.RG_VARIANT_SMALLT, inputs.Q8_0, A, 60, 256, A, 1, A, 0.0) == rg.RG_ERR_SHAPE
    # the named small-T route: rows TMA cannot address (Q6_K at K = 256), or
    # more rows of X than its grid holds, are shape errors before any launch
    assert rg.rg_mul_mat_variant(rg.RG_VARIANT_SMALLT, inputs.Q6_K, A, 64, 256, A, 1, A, 0.0) == rg.RG_ERR_SHAPE
    assert rg.rg_mul_mat_variant(rg.RG_VARIANT_SMALLT, inputs.Q8_0, A, 64, 256, A, 4 * 65535 + 1, A,
                                 0.0) == rg.RG_ERR_SHAPE
    # one or two rows of X with aligned rows take no workspace
    for T in (1, 2):
        assert rg.rg_mul_mat_workspace_bytes(inputs.Q4_K, 14336, 4096, T) == 0


def test_out_prod_lora_validation(lib):
    """The adapter entry checks its own arguments after the base product's."""
    A = 0x1000
    base = (0, inputs.Q8_0, A, 64, 256, A, 8, A, 0.0)

    def call(*args, a=A, b=A, rank=16, scale=1.0, prefix=base):
        return rg.rg_out_prod_lora(*prefix, a, b, rank, scale)
    assert call(rank=-1) == rg.RG_ERR_ARG
    assert call(rank=1025) == rg.RG_ERR_SHAPE
    assert call(a=None) == rg.RG_ERR_ARG
    assert call(b=None) == rg.RG_ERR_ARG
    assert call(a=A + 4) == rg.RG_ERR_ALIGN
    assert call(b=A + 8) == rg.RG_ERR_ALIGN
    assert call(prefix=(9, inputs.Q8_0, A, 64, 256, A, 8, A, 0.0)) == rg.RG_ERR_TYPE
    assert call(prefix=(0, 16, A, 64, 256, A, 8, A, 0.0)) == rg.RG_ERR_TYPE
    assert call(prefix=(0, inputs.Q8_0, A, 64, 200, A, 8, A, 0.0)) == rg.RG_ERR_SHAPE
    # nothing to compute: T == 0 or K == 0, whatever the adapter pointers
    assert call(a=None, b=None, prefix=(0, inputs.Q8_0, None, 64, 256, None, 0, None, 0.0)) == rg.RG_OK
    assert call(a=None, b=None, prefix=(0, inputs.Q8_0, None, 64, 0, None, 8, None, 0.0)) == rg.RG_OK
