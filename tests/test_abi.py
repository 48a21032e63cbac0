"""Host-side checks of the C ABI, no GPU needed: the library builds, loads and
exports every function include/fa.h declares; the pure host functions answer;
argument errors come back as status codes before any device work."""
import ctypes
import os
import re
import subprocess

import pytest

import exact_attention_97_gb300 as fa
from exact_attention_97_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ["fa_fwd", "fa_bwd", "fa_fwd_f32", "fa_bwd_f32", "fa_bwd_workspace_size",
              "fa_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (fa_[a-z0-9_]+)", out))
    for name in _declared():
        assert name in exported, name
        assert getattr(lib, name) is not None
    assert set(_declared()) <= set(_lib._SIGNATURES)


def test_status_strings(lib):
    for code in range(10):
        s = fa.fa_status_string(code)
        assert s and s != "unknown status"
    assert fa.fa_status_string(1234) == "unknown status"


def test_workspace_size_layout():
    # bf16: padded L and D rows (B*H*ceil(N/128)*128 fp32 each)
    def r256(x):
        return (x + 255) // 256 * 256
    for B, H, N, d in [(1, 1, 1, 64), (2, 3, 300, 128), (8, 32, 4096, 128), (1, 32, 65536, 128)]:
        prow = B * H * ((N + 127) // 128 * 128)
        want = 2 * r256(prow * 4)
        assert fa.fa_bwd_workspace_size(B, H, N, d, fa.FA_BF16) == want
        assert fa.fa_bwd_workspace_size(B, H, N, d, fa.FA_F32) == r256(B * H * N * 4)
        assert fa.fa_bwd_workspace_size(B, H, N, d, fa.FA_F16) == want
    assert fa.fa_bwd_workspace_size(0, 1, 1, 64, fa.FA_BF16) == 0
    assert fa.fa_bwd_workspace_size(1, 1, 1, 129, fa.FA_BF16) == 0
    assert fa.fa_bwd_workspace_size(1, 1, 1, 64, 7) == 0


P = 0x10000  # a fake, 16-byte aligned "device pointer": never dereferenced, validation fails first


def _fwd(lib, q=P, k=P, v=P, o=P, lse=P, B=1, H=1, N=128, d=64, scale=0.125, causal=0):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, None)


def _bwd(lib, ws=P, ws_bytes=1 << 40, B=1, H=1, N=128, d=64, scale=0.125, ptr=P, **kw):
    ptrs = [kw.get(n, ptr) for n in ("q", "k", "v", "o", "lse", "dO", "dq", "dk", "dv")]
    return lib.fa_bwd(*ptrs, B, H, N, d, scale, 0, ws, ws_bytes, None)


def test_fwd_argument_errors(lib):
    assert _fwd(lib, q=None) == 1
    assert _fwd(lib, lse=None) == 1
    assert _fwd(lib, N=0) == 2
    assert _fwd(lib, B=-1) == 2
    assert _fwd(lib, d=0) == 2
    assert _fwd(lib, d=512) == 2
    assert _fwd(lib, d=80) == 3          # valid head size without a bf16 kernel
    assert _fwd(lib, d=200) == 3
    assert _fwd(lib, B=300, H=300) == 3  # more than 65535 heads
    assert _fwd(lib, N=1 << 30, B=4, H=4, d=128) == 2  # 2^40 elements
    assert _fwd(lib, q=P + 8) == 4       # TMA needs 16-byte aligned bases
    assert _fwd(lib, lse=P + 2) == 4
    assert _fwd(lib, scale=float("nan")) == 9
    assert _fwd(lib, scale=float("inf")) == 9


def test_bwd_argument_errors(lib):
    assert _bwd(lib, dk=None) == 1
    assert _bwd(lib, N=-3) == 2
    assert _bwd(lib, d=80) == 3
    assert _bwd(lib, d=256) == 3  # the d = 256 kernel is forward only
    assert _bwd(lib, d=512) == 2
    assert _bwd(lib, dv=P + 4) == 4
    assert _bwd(lib, ws=None) == 5
    need = fa.fa_bwd_workspace_size(1, 1, 128, 64, fa.FA_BF16)
    assert _bwd(lib, ws_bytes=need - 1) == 5
    assert _bwd(lib, ws=P + 16, ws_bytes=need) == 4  # workspace must be 256-byte aligned
    assert _bwd(lib, scale=float("-inf")) == 9


def test_f16_argument_errors(lib):
    args = [P] * 5
    assert lib.fa_fwd_f16(None, *args[1:], 1, 1, 128, 64, 0.125, 0, None) == 1
    assert lib.fa_fwd_f16(*args, 1, 1, 128, 80, 0.125, 0, None) == 3
    assert lib.fa_fwd_f16(P + 8, *args[1:], 1, 1, 128, 64, 0.125, 0, None) == 4
    ptrs = [P] * 9
    assert lib.fa_bwd_f16(*ptrs, 1, 1, 128, 64, 0.125, 0, None, 0, None) == 5
    assert lib.fa_bwd_f16(*ptrs, 1, 1, 128, 64, float("nan"), 0, P, 1 << 30, None) == 9


def test_dropout_argument_errors(lib):
    args = [P] * 5
    for bad in (1.0, 1.5, -0.1, float("nan"), float("inf")):
        assert lib.fa_fwd_dropout(*args, 1, 1, 128, 128, 64, 0.125, 0, fa.FA_BF16, bad, 1, 0, 0, None) == 9
    assert lib.fa_fwd_dropout(*args, 1, 1, 128, 128, 64, 0.125, 0, fa.FA_F32, 0.1, 1, 0, 0, None) == 3
    assert lib.fa_fwd_dropout(None, *args[1:], 1, 1, 128, 128, 64, 0.125, 0, fa.FA_BF16, 0.1, 1, 0, 0, None) == 1
    assert lib.fa_fwd_dropout(*args, 1, 1, 128, 128, 80, 0.125, 0, fa.FA_F16, 0.1, 1, 0, 0, None) == 3
    ptrs = [P] * 9
    assert lib.fa_bwd_dropout(*ptrs, 1, 1, 128, 128, 64, 0.125, 0, fa.FA_BF16, 1.0, 1, 0, 0, P, 1 << 30, None) == 9
    assert lib.fa_bwd_dropout(*ptrs, 1, 1, 128, 128, 64, 0.125, 0, fa.FA_BF16, 0.2, 1, 0, 0, None, 0, None) == 5
    assert lib.fa_bwd_dropout(*ptrs, 1, 1, 128, 128, 256, 0.125, 0, fa.FA_BF16, 0.2, 1, 0, 0, P, 1 << 30,
                              None) == 3


def test_kv_argument_errors(lib):
    args = [P] * 5
    # causal with fewer keys than queries: the leading queries would see nothing
    assert lib.fa_fwd_kv(*args, 1, 1, 300, 200, 64, 0.125, 1, fa.FA_BF16, None) == 2
    assert lib.fa_fwd_kv(*args, 1, 1, 300, 0, 64, 0.125, 0, fa.FA_BF16, None) == 2
    assert lib.fa_fwd_kv(*args, 1, 1, 300, 200, 64, 0.125, 0, fa.FA_F32, None) == 3
    assert lib.fa_fwd_kv(*args, 1, 1, 300, 200, 64, 0.125, 0, 7, None) == 9
    ptrs = [P] * 9
    assert lib.fa_bwd_kv(*ptrs, 1, 1, 100, 64, 64, 0.125, 1, fa.FA_F16, P, 1 << 30, None) == 2
    need = fa.fa_bwd_workspace_size(1, 1, 100, 64, fa.FA_F16)
    assert lib.fa_bwd_kv(*ptrs, 1, 1, 100, 640, 64, 0.125, 1, fa.FA_F16, P, need - 16, None) == 5


def test_f32_argument_errors(lib):
    args = [P] * 5
    assert lib.fa_fwd_f32(None, *args[1:], 1, 1, 4, 2, 1.0, 0, None) == 1
    assert lib.fa_fwd_f32(*args, 1, 1, 4, 129, 1.0, 0, None) == 2
    assert lib.fa_fwd_f32(P + 2, *args[1:], 1, 1, 4, 2, 1.0, 0, None) == 4
    ptrs = [P] * 9
    assert lib.fa_bwd_f32(*ptrs, 1, 1, 4, 2, 1.0, 0, None, 0, None) == 5


def test_dropout_workspace_size():
    """The shared-bits workspace is the plain one followed by the saved-bits
    layout; shapes and types the dropout backward rejects give 0."""
    for B, H, Nq, Nk, d in [(1, 1, 1, 1, 64), (2, 3, 300, 513, 96), (8, 32, 4096, 4096, 128), (64, 32, 128, 8192, 128)]:
        for kind in (fa.FA_BF16, fa.FA_F16):
            want = fa.fa_bwd_workspace_size(B, H, Nq, d, kind) + fa.fa_dropout_mask_size(B, H, Nq, Nk)
            assert fa.fa_bwd_dropout_workspace_size(B, H, Nq, Nk, d, kind) == want
    assert fa.fa_bwd_workspace_size(2, 3, 300, 96, fa.FA_BF16) % 256 == 0  # the bits start 256-byte aligned
    assert fa.fa_bwd_dropout_workspace_size(1, 1, 128, 128, 64, fa.FA_F32) == 0
    assert fa.fa_bwd_dropout_workspace_size(1, 1, 128, 128, 256, fa.FA_BF16) == 0
    assert fa.fa_bwd_dropout_workspace_size(1, 1, 128, 128, 80, fa.FA_BF16) == 0
    assert fa.fa_bwd_dropout_workspace_size(0, 1, 128, 128, 64, fa.FA_BF16) == 0
    assert fa.fa_bwd_dropout_workspace_size(1, 1, 128, 0, 64, fa.FA_BF16) == 0


def test_dropout_mask_size_and_argument_errors(lib):
    assert fa.fa_dropout_mask_size(8, 32, 4096, 4096) == 8 * 32 * 32 * 32 * 2048
    assert fa.fa_dropout_mask_size(1, 2, 300, 129) == 2 * 3 * 2 * 2048
    assert fa.fa_dropout_mask_size(0, 1, 1, 1) == 0
    need = fa.fa_dropout_mask_size(1, 1, 128, 128)
    args = [P] * 5
    fwd = lambda mask, nbytes, p=0.1, Nq=128: lib.fa_fwd_dropout_mask(  # noqa: E731
        *args, 1, 1, Nq, 128, 64, 0.125, 0, fa.FA_BF16, p, 1, 0, 0, mask, nbytes, None)
    assert fwd(None, need) == 1
    assert fwd(P + 8, need) == 4
    assert fwd(P, need - 16) == 5
    assert fwd(P, need, p=1.0) == 9
    assert fwd(P, need, Nq=0) == 2
    ptrs = [P] * 9
    bwd = lambda mask, nbytes: lib.fa_bwd_dropout_mask(  # noqa: E731
        *ptrs, 1, 1, 128, 128, 64, 0.125, 0, fa.FA_BF16, 0.1, mask, nbytes, P, 1 << 30, None)
    assert bwd(None, need) == 1
    assert bwd(P, need - 1) == 5


def test_status_read_argument_errors(lib):
    assert lib.fa_status_async(None, None) == 1
    assert lib.fa_status_async(P + 2, None) == 4
    assert lib.fa_status_word(None) == 1


def test_no_cpu_fallback_in_the_binding():
    """The binding only marshals arguments: it never imports the oracle or
    computes attention itself."""
    import ast
    bad_calls = {"softmax", "matmul", "einsum", "bmm", "mm", "scaled_dot_product_attention", "exp"}
    pkg = os.path.join(ROOT, "exact_attention_97_gb300")
    for fn in os.listdir(pkg):
        if not fn.endswith(".py"):
            continue
        tree = ast.parse(open(os.path.join(pkg, fn)).read())
        for node in ast.walk(tree):
            if isinstance(node, ast.Import):
                assert not any(a.name.split(".")[0] == "oracle" for a in node.names), fn
            if isinstance(node, ast.ImportFrom):
                assert (node.module or "").split(".")[0] != "oracle", fn
            if isinstance(node, ast.Call):
                f = node.func
                name = f.attr if isinstance(f, ast.Attribute) else getattr(f, "id", "")
                assert name not in bad_calls, (fn, name)
            if isinstance(node, ast.BinOp):
                assert not isinstance(node.op, ast.MatMult), fn
