"""The C-ABI library loads, exports every declared symbol and validates arguments.

CPU only: nothing here reaches a device.  Every call below fails validation
before any CUDA call, so it returns without a GPU.
"""

import os
import re
import subprocess

import pytest

import exact_io_aware_31_gb300 as fa
from exact_io_aware_31_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(fa.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fa.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s(fa_[a-z0-9_]+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "fa.h"\nint main(void){ return (int)sizeof(&fa_fwd) == 0; }\n')
    cuda_inc = "/usr/local/cuda/include"
    r = subprocess.run(["gcc", "-std=c99", "-fsyntax-only", "-I", os.path.dirname(HEADER), "-I", cuda_inc, str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_status_strings(lib):
    names = ["FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_WORKSPACE", "FA_ERR_CUDA",
             "FA_ERR_DEVICE_TIMEOUT", "FA_ERR_INTERNAL"]
    for code, name in enumerate(names):
        assert fa.fa_status_string(code).startswith(name)
    assert fa.fa_status_string(99) == "unknown fa status"
    assert fa.fa_status_string(-1) == "unknown fa status"


def test_workspace_size(lib):
    # fp32 dQ accumulator [B,H,N,d] + two fp32 row arrays [B,H,Npad], each 256-byte aligned
    def expect(B, H, N, d):
        r = lambda x: (x + 255) // 256 * 256
        npad = (N + 127) // 128 * 128
        return r(B * H * N * d * 4) + 2 * r(B * H * npad * 4)
    for args in [(1, 2, 256, 64), (64, 16, 1024, 64), (1, 16, 16384, 128), (1, 1, 1, 128), (3, 5, 1000, 64)]:
        assert fa.fa_bwd_workspace_size(*args) == expect(*args)
    assert fa.fa_bwd_workspace_size(1, 1, 16, 96) == 0
    assert fa.fa_bwd_workspace_size(0, 1, 16, 64) == 0
    assert fa.fa_bwd_workspace_size(1, 1, 0, 64) == 0


A = 1 << 20  # a 16-byte aligned fake address; validation fails before it is used


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=-1), fa.FA_ERR_INVALID_ARG),
    (dict(N=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED),
    (dict(causal=2), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(o=A + 8), fa.FA_ERR_INVALID_ARG),
    (dict(lse=A + 4), fa.FA_ERR_INVALID_ARG),
    (dict(B=1 << 16, H=1 << 16), fa.FA_ERR_INVALID_ARG),
])
def test_fwd_validation(lib, kw, code):
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=1, N=16, d=64, scale=0.125, causal=0, stream=None)
    args.update(kw)
    assert fa.fa_fwd(**args) == code


@pytest.mark.parametrize("kw,code", [
    (dict(N=-5), fa.FA_ERR_INVALID_ARG),
    (dict(d=32), fa.FA_ERR_UNSUPPORTED),
    (dict(dout=A + 2), fa.FA_ERR_INVALID_ARG),
    (dict(dk=None), fa.FA_ERR_INVALID_ARG),
    (dict(workspace=None), fa.FA_ERR_WORKSPACE),
    (dict(workspace=A + 16), fa.FA_ERR_WORKSPACE),
    (dict(workspace_bytes=100), fa.FA_ERR_WORKSPACE),
])
def test_bwd_validation(lib, kw, code):
    args = dict(q=A, k=A, v=A, o=A, dout=A, lse=A, dq=A, dk=A, dv=A, B=1, H=1, N=16, d=64, scale=0.125,
                causal=1, workspace=A, workspace_bytes=1 << 30, stream=None)
    args.update(kw)
    assert fa.fa_bwd(**args) == code


def test_tensor_helpers_reject_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.forward(q, q, q)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nq=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nk=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nq=9), fa.FA_ERR_UNSUPPORTED),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(Nq=4, Nk=3, causal=1), fa.FA_ERR_INVALID_ARG),
    (dict(num_splits=-1), fa.FA_ERR_INVALID_ARG),
    (dict(causal=3), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(q=A + 2), fa.FA_ERR_INVALID_ARG),
    (dict(lse=None), fa.FA_ERR_INVALID_ARG),
])
def test_splitkv_validation(lib, kw, code):
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=2, Nq=1, Nk=1000, d=128, scale=0.1, causal=1, num_splits=0,
                workspace=None, workspace_bytes=0, stream=None)
    args.update(kw)
    assert fa.fa_fwd_splitkv(**args) == code


def test_splitkv_workspace_size_of_invalid_sizes_is_zero(lib):
    assert fa.fa_fwd_splitkv_workspace_size(1, 1, 9, 100, 64, 0) == 0     # Nq > 8
    assert fa.fa_fwd_splitkv_workspace_size(1, 1, 1, 100, 96, 0) == 0     # d = 96
    assert fa.fa_fwd_splitkv_workspace_size(0, 1, 1, 100, 64, 0) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(dq=None), fa.FA_ERR_INVALID_ARG),
    (dict(workspace=None), fa.FA_ERR_WORKSPACE),
])
def test_bwd_deterministic_validation(lib, kw, code):
    args = dict(q=A, k=A, v=A, o=A, dout=A, lse=A, dq=A, dk=A, dv=A, B=1, H=1, N=16, d=64, scale=0.125,
                causal=1, workspace=A, workspace_bytes=1 << 30, stream=None)
    args.update(kw)
    assert fa.fa_bwd_deterministic(**args) == code


@pytest.mark.parametrize("p", [-0.1, 1.0, 1.5, float("nan")])
def test_dropout_rate_validation(lib, p):
    assert fa.fa_fwd_dropout(A, A, A, A, A, 1, 1, 16, 64, 0.125, 0, p, 1, 0, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_dropout(A, A, A, A, A, A, A, A, A, 1, 1, 16, 64, 0.125, 0, p, 1, 0, A, 1 << 30,
                             None) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,code", [
    (dict(d=64), fa.FA_ERR_UNSUPPORTED),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(N=0), fa.FA_ERR_INVALID_ARG),
    (dict(causal=2), fa.FA_ERR_INVALID_ARG),
    (dict(q_descale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-0.125), fa.FA_ERR_INVALID_ARG),      # the E4M3 path takes no negative scale
    (dict(k_descale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(k_descale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(q_descale=3e38, k_descale=3e38), fa.FA_ERR_INVALID_ARG),   # product with scale overflows
    (dict(q8=A + 8), fa.FA_ERR_INVALID_ARG),
    (dict(v=None), fa.FA_ERR_INVALID_ARG),
])
def test_fwd_fp8_validation(lib, kw, code):
    args = dict(q8=A, k8=A, v=A, o=A, lse=A, B=1, H=1, N=16, d=128, scale=0.125, q_descale=1.0, k_descale=1.0,
                causal=0, stream=None)
    args.update(kw)
    assert fa.fa_fwd_fp8(**args) == code


def test_fp8_helper_rejects_cpu_tensors(lib):
    import torch
    q8 = torch.zeros(1, 1, 8, 128, dtype=torch.uint8)
    v = torch.zeros(1, 1, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.forward_fp8(q8, q8, v)


@pytest.mark.parametrize("kw,code", [
    (dict(d=32), fa.FA_ERR_UNSUPPORTED),
    (dict(N=0), fa.FA_ERR_INVALID_ARG),
    (dict(o=A + 4), fa.FA_ERR_INVALID_ARG),
    (dict(lse=None), fa.FA_ERR_INVALID_ARG),
    (dict(workspace=None), fa.FA_ERR_WORKSPACE),
    (dict(workspace_bytes=1024), fa.FA_ERR_WORKSPACE),
])
def test_bwd_preprocess_validation(lib, kw, code):
    args = dict(o=A, dout=A, lse=A, B=1, H=1, N=16, d=64, workspace=A, workspace_bytes=1 << 30, stream=None)
    args.update(kw)
    assert fa.fa_bwd_preprocess(**args) == code


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(causal=5), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(dv=A + 8), fa.FA_ERR_INVALID_ARG),
    (dict(dout=None), fa.FA_ERR_INVALID_ARG),
    (dict(workspace=A + 128), fa.FA_ERR_WORKSPACE),
])
def test_bwd_dkdv_validation(lib, kw, code):
    args = dict(q=A, k=A, v=A, dout=A, dk=A, dv=A, B=1, H=1, N=16, d=64, scale=0.125, causal=1, workspace=A,
                workspace_bytes=1 << 30, stream=None)
    args.update(kw)
    assert fa.fa_bwd_dkdv(**args) == code


@pytest.mark.parametrize("kw,code", [
    (dict(d=256), fa.FA_ERR_UNSUPPORTED),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(dq=A + 2), fa.FA_ERR_INVALID_ARG),
    (dict(workspace=None), fa.FA_ERR_WORKSPACE),
])
def test_bwd_dq_convert_validation(lib, kw, code):
    args = dict(dq=A, B=1, H=1, N=16, d=64, scale=0.125, workspace=A, workspace_bytes=1 << 30, stream=None)
    args.update(kw)
    assert fa.fa_bwd_dq_convert(**args) == code


# Oversized for the 64 MiB scratch of fa_bwd_noalloc (a 128 MiB dQ accumulator).
BIG = dict(B=1, H=64, N=4096, d=128)


@pytest.mark.parametrize("kw,code", [
    (dict(), fa.FA_ERR_WORKSPACE),                        # valid, too large: refused before any device work
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),    # bad arguments are named as such, whatever the size
    (dict(scale=-1.0), fa.FA_ERR_WORKSPACE),              # a negative scale is valid
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(causal=2), fa.FA_ERR_INVALID_ARG),
    (dict(dq=A + 4), fa.FA_ERR_INVALID_ARG),
    (dict(lse=None), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(B=1, H=1, N=16, d=96), fa.FA_ERR_UNSUPPORTED),
])
def test_noalloc_validates_arguments_before_its_size_limit(lib, kw, code):
    args = dict(q=A, k=A, v=A, o=A, dout=A, lse=A, dq=A, dk=A, dv=A, **BIG, scale=0.1, causal=0, stream=None)
    args.update(kw)
    assert fa.fa_bwd_noalloc(**args) == code


def test_noalloc_limit_is_the_workspace_size(lib):
    """B2 H8 N8064 d128 fits the 64 MiB scratch (16 KiB to spare); one more row does not (refused on the CPU)."""
    assert fa.NOALLOC_SCRATCH_BYTES - (16 << 10) == fa.fa_bwd_workspace_size(2, 8, 8064, 128)
    assert fa.fa_bwd_workspace_size(2, 8, 8065, 128) > fa.NOALLOC_SCRATCH_BYTES
    args = dict(q=A, k=A, v=A, o=A, dout=A, lse=A, dq=A, dk=A, dv=A, B=2, H=8, N=8065, d=128, scale=0.1, causal=1,
                stream=None)
    assert fa.fa_bwd_noalloc(**args) == fa.FA_ERR_WORKSPACE
