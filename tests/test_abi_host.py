"""Host-side checks of the C-ABI library, no GPU needed: it loads, exports
every function include/tpmlp.h declares, and rejects bad arguments with the
documented status before touching the device (so no call here reaches CUDA).
"""

import ctypes
import os
import re

import pytest

from tensor_transformer_mlp_columnparallel_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return B.lib()


@pytest.fixture(autouse=True)
def no_launch(request):
    """Every rejected call returns before any kernel launch."""
    if "lib" not in request.fixturenames:
        yield
        return
    before = B.lib().tpmlp_launch_count()
    yield
    assert B.lib().tpmlp_launch_count() == before


PP = ctypes.POINTER(ctypes.c_void_p)


def ptrs(*vals):
    arr = (ctypes.c_void_p * len(vals))(*vals)
    return ctypes.cast(arr, PP)


FAKE = 0x10000   # a 16-byte-aligned address that is never dereferenced


def fwd(lib, dt=1, N=4, D=16, F=32, T=2, act=1, X=FAKE, W1="ok", b1=None, W2="ok", b2=None,
        Y=FAKE, H="ok", Z=None, mode=1, ws=None, ws_bytes=0):
    sh = lambda v: ptrs(*([FAKE] * T)) if v == "ok" else v
    return lib.tpmlp_forward(dt, N, D, F, T, act, X, sh(W1), b1, sh(W2), b2, Y, sh(H), Z, mode, ws,
                             ws_bytes, None)


def test_library_exports_every_declared_function(lib):
    names = B.header_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    # and the binding wraps each one under the same name
    import tensor_transformer_mlp_columnparallel_gb300 as tp
    for n in names:
        if n == "tpmlp_status_str":
            continue
        assert hasattr(tp._binding, n), n


def test_status_strings(lib):
    for s in range(8):
        assert B.status_str(s).startswith("TPMLP_")
    assert "unknown" in B.status_str(99)


def test_workspace_bytes(lib):
    import torch
    r256 = lambda x: (x + 255) // 256 * 256
    N, D, F, T = 100, 24, 64, 4
    assert B.tpmlp_workspace_bytes(0, torch.bfloat16, N, D, F, T, "splitk") == 0
    assert B.tpmlp_workspace_bytes(0, torch.bfloat16, N, D, F, T, "partials") == T * r256(N * D * 4)
    assert B.tpmlp_workspace_bytes(1, torch.bfloat16, N, D, F, T, "splitk") == T * r256(N * (F // T) * 2)
    assert B.tpmlp_workspace_bytes(1, torch.float32, N, D, F, T, "partials") == \
        T * r256(N * (F // T) * 4) + T * r256(N * D * 4)
    assert lib.tpmlp_workspace_bytes(0, 1, N, D, 63, 4, 0) == ctypes.c_size_t(-1).value


def test_workspace_bytes_balanced(lib):
    """The balanced size adds the GEMMs' stream-K scratch (bf16, N >= 1) after
    the required part rounded to 256 bytes. For 1 <= N <= 64: 4 counters per
    128-column tile of the widest GEMM (T groups of max(F/T, D) columns), then
    min(256, units) CTAs x 2 slots x round_up(N, 32) rows x 256 fp32 columns,
    units = T x max(ceil(F/T / 128) ceil(D / 64), ceil(D / 128) ceil(F/T / 64)),
    the (tile, k-block) units of the block's GEMMs. For N > 64 (the part wave
    only): 256 x 8 counters, then 256 CTAs x 2 slots x 128 rows x 256 fp32
    columns (64 MiB)."""
    import torch
    r256 = lambda x: (x + 255) // 256 * 256
    cdiv = lambda a, b: -(-a // b)
    bal = B.tpmlp_workspace_bytes_balanced
    for D, F, T in ((1024, 8192, 4), (256, 1024, 2), (2048, 24, 3)):
        Fs = F // T
        units = T * max(cdiv(Fs, 128) * cdiv(D, 64), cdiv(D, 128) * cdiv(Fs, 64))
        for N in (1, 16, 33, 64, 65, 4096):
            if N <= 64:
                rows = (N + 31) // 32 * 32
                sk = r256(4 * T * cdiv(max(Fs, D), 128) * 4) + min(256, units) * 2 * rows * 256 * 4
            else:
                sk = r256(256 * 8 * 4) + 256 * 2 * 128 * 256 * 4
            for op in (0, 1):
                for mode in ("splitk", "partials"):
                    base = B.tpmlp_workspace_bytes(op, torch.bfloat16, N, D, F, T, mode)
                    assert bal(op, torch.bfloat16, N, D, F, T, mode) == r256(base) + sk
    D, F, T = 1024, 8192, 4
    # no scratch for fp32 and for N = 0
    for args in ((torch.float32, 16), (torch.float32, 4096), (torch.bfloat16, 0)):
        for mode in ("splitk", "partials"):
            assert bal(0, args[0], args[1], D, F, T, mode) == \
                B.tpmlp_workspace_bytes(0, args[0], args[1], D, F, T, mode)
    assert lib.tpmlp_workspace_bytes_balanced(0, 1, 16, D, 63, 4, 0) == ctypes.c_size_t(-1).value


def test_shape_errors(lib):
    assert fwd(lib, F=33, T=2) == B.ERR_SHAPE             # F % T != 0 (the pages' assert)
    assert fwd(lib, T=0) == B.ERR_SHAPE
    assert fwd(lib, T=17, F=17 * 8) == B.ERR_SHAPE
    assert fwd(lib, D=0) == B.ERR_SHAPE
    assert fwd(lib, N=-1) == B.ERR_ARG


def test_enum_errors(lib):
    assert fwd(lib, dt=7) == B.ERR_DTYPE
    assert fwd(lib, act=5) == B.ERR_ARG
    assert fwd(lib, mode=9) == B.ERR_ARG


def test_pointer_and_alignment_errors(lib):
    assert fwd(lib, X=None) == B.ERR_ARG
    assert fwd(lib, W1=None) == B.ERR_ARG
    assert fwd(lib, W1=ptrs(FAKE, None)) == B.ERR_ARG
    assert fwd(lib, X=FAKE + 2) == B.ERR_ALIGN            # bf16 tensor-memory-access rule
    assert fwd(lib, H=ptrs(FAKE, FAKE + 8)) == B.ERR_ALIGN
    assert fwd(lib, D=12) == B.ERR_ALIGN                  # row pitch of 24 bytes
    assert fwd(lib, F=2 * 12) == B.ERR_ALIGN              # F/T = 12
    # the fp32 CUDA-core path has no alignment rule, so the same odd shapes
    # only fail on the (absent) pointers
    assert fwd(lib, dt=0, D=12, X=None) == B.ERR_ARG


def test_workspace_errors(lib):
    assert fwd(lib, mode=0) == B.ERR_WORKSPACE            # PARTIALS needs a workspace
    assert fwd(lib, mode=0, ws=FAKE, ws_bytes=10) == B.ERR_WORKSPACE
    assert lib.tpmlp_backward(1, 4, 16, 32, 2, 1, FAKE, ptrs(FAKE, FAKE), ptrs(FAKE, FAKE),
                              ptrs(FAKE, FAKE), ptrs(FAKE, FAKE), FAKE, FAKE, ptrs(FAKE, FAKE),
                              ptrs(FAKE, FAKE), None, None, 1, None, 0, None) == B.ERR_WORKSPACE


def test_empty_batch_forward_is_a_no_op(lib):
    assert fwd(lib, N=0, X=None, Y=None, H=None) == B.OK


def test_vocab_ce_and_reduce_errors(lib):
    assert lib.tpmlp_vocab_ce(4, 10, 3, FAKE, FAKE, FAKE, None, None, None, None) == B.ERR_SHAPE
    assert lib.tpmlp_vocab_ce(4, 12, 0, FAKE, FAKE, FAKE, None, None, None, None) == B.ERR_SHAPE
    assert lib.tpmlp_vocab_ce(4, 12, 3, None, FAKE, FAKE, None, None, None, None) == B.ERR_ARG
    assert lib.tpmlp_block_reduce(1, 4, 8, 2, ptrs(FAKE, None), None, FAKE, None) == B.ERR_ARG
    assert lib.tpmlp_block_reduce(3, 4, 8, 2, ptrs(FAKE, FAKE), None, FAKE, None) == B.ERR_DTYPE


def test_gemm_plan_argument_errors(lib):
    x = ctypes.c_int(0)
    r = ctypes.byref(x)
    for bal in (0, 1):
        assert lib.tpmlp_gemm_plan(16, 128, 64, 1, 0, 0, bal, None, r, r) == B.ERR_ARG
        assert lib.tpmlp_gemm_plan(0, 128, 64, 1, 0, 0, bal, r, r, r) == B.ERR_SHAPE
        assert lib.tpmlp_gemm_plan(16, 128, 64, 0, 0, 0, bal, r, r, r) == B.ERR_SHAPE
        assert lib.tpmlp_gemm_plan(16, 128, 64, 17, 1, 0, bal, r, r, r) == B.ERR_SHAPE
        assert lib.tpmlp_gemm_plan(1 << 31, 128, 64, 1, 0, 0, bal, r, r, r) == B.ERR_SHAPE


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(ImportError):
        B.lib()


def test_product_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "tensor_transformer_mlp_columnparallel_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
                assert "oracle/" not in src, f


def test_gemm_stall_self_test_role_is_checked(lib):
    assert lib.tpmlp_selftest_gemm_stall(4) == B.ERR_ARG
    assert lib.tpmlp_selftest_gemm_stall(-1) == B.ERR_ARG
    for role in (1, 2, 3, 0):
        assert lib.tpmlp_selftest_gemm_stall(role) == B.OK


def test_every_environment_switch_is_documented_in_the_header():
    """The library's sources read only environment variables that the public
    header describes (launch-order switches that never change results)."""
    csrc = os.path.join(ROOT, "tensor_transformer_mlp_columnparallel_gb300", "csrc")
    names = set()
    for f in os.listdir(csrc):
        if f.endswith((".cu", ".cuh", ".h", ".cpp")):
            names |= set(re.findall(r'getenv\("([A-Z0-9_]+)"\)', open(os.path.join(csrc, f)).read()))
    assert names, "no environment switches found"
    header = open(os.path.join(ROOT, "include", "tpmlp.h")).read()
    for n in sorted(names):
        assert n in header, n
