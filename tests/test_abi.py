"""Host-side checks of the C ABI that need no GPU: the library builds/loads,
exports every entry point include/jetfp8.h declares, and the binding knows
each one's arity."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "jetfp8.h")


def _declared():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(jetfp8_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from fp8_mixed_granularity_gb300 import jetfp8
    return jetfp8.load_library()


def test_header_declares_the_hot_path():
    names = _declared()
    for n in ["jetfp8_quant_act_1x128", "jetfp8_quant_weight_128x128",
              "jetfp8_requant_rowgrp_to_colgrp", "jetfp8_quant_grad_dual",
              "jetfp8_rmsnorm_quant", "jetfp8_gemm_fprop", "jetfp8_gemm_dgrad",
              "jetfp8_gemm_wgrad"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    from fp8_mixed_granularity_gb300 import jetfp8
    # entry points that return something other than a status are bound apart
    not_status = {"jetfp8_status_string", "jetfp8_rmsnorm_bwd_workspace_bytes", "jetfp8_nvfp4_scale_bytes"}
    for name in _declared():
        if name not in not_status:
            assert name in jetfp8.SIGNATURES, name
        if name != "jetfp8_status_string":
            assert callable(getattr(jetfp8, name)), name


def test_status_strings(lib):
    for code, text in [(0, b"JETFP8_OK"), (2, b"JETFP8_ERR_UNSUPPORTED_SHAPE"), (5, b"JETFP8_ERR_TIMEOUT")]:
        assert lib.jetfp8_status_string(code) == text


def test_validation_rejects_before_touching_the_device(lib):
    """Null pointers and bad shapes are refused synchronously, before any
    CUDA call (so this runs on a machine without a GPU)."""
    P = ctypes.c_void_p
    # null input
    assert lib.jetfp8_quant_act_1x128(None, 4, 128, P(64), P(64), None) == 1
    # K not a multiple of 128
    assert lib.jetfp8_quant_act_1x128(P(64), 4, 100, P(64), P(64), None) == 2
    # misaligned pointer
    assert lib.jetfp8_quant_act_1x128(P(48), 4, 128, P(64), P(64), None) == 3   # bf16 needs 32 B
    assert lib.jetfp8_quant_act_1x128(P(64), 4, 128, P(72), P(64), None) == 3   # E4M3 needs 16 B
    # fused output quantiser: the output width must be a multiple of 256
    assert lib.jetfp8_gemm_fprop_quant(P(64), P(64), P(64), P(64), 4, 384, 128, None, P(64), P(64), None) == 2
    assert lib.jetfp8_gemm_dgrad_quant(P(64), P(64), P(64), P(64), 4, 256, 384, None, P(64), P(64), None) == 2
    # RMSNorm backward: workspace size and a too-small workspace
    lib.jetfp8_rmsnorm_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.jetfp8_rmsnorm_bwd_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    # rows up to 4096 wide: one workspace row per CTA of 8 warps (at most 152 CTAs)
    assert lib.jetfp8_rmsnorm_bwd_workspace_bytes(300, 256) == 38 * 256 * 4
    assert lib.jetfp8_rmsnorm_bwd_workspace_bytes(100000, 4096) == 152 * 4096 * 4
    # wider rows: one workspace row per 128-row chunk
    assert lib.jetfp8_rmsnorm_bwd_workspace_bytes(300, 8192) == 3 * 8192 * 4
    assert lib.jetfp8_rmsnorm_bwd(P(64), P(64), P(64), P(64), ctypes.c_int64(300), ctypes.c_int64(256),
                                  P(64), P(64), P(64), ctypes.c_size_t(38 * 256 * 4 - 4), None) == 1
    # WGrad needs M multiple of 128
    assert lib.jetfp8_gemm_wgrad(P(64), P(64), P(64), P(64), 100, 128, 128, P(64), 0, None) == 2
    # non-positive M
    assert lib.jetfp8_gemm_fprop(P(64), P(64), P(64), P(64), 0, 128, 128, P(64), 0, None) == 1


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="passes placeholder addresses: only where no GPU can be reached")
def test_noalloc_rejects_scratch_above_8mib(lib):
    """The allocation-free RMSNorm backward refuses sizes whose scratch would
    exceed its fixed 8 MiB.  Placeholder (never dereferenced) addresses are
    passed, so this runs only on a machine without a GPU: there, even if the
    size check were skipped, the device check after it would refuse the call
    before any launch."""
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    fn = lib.jetfp8_rmsnorm_bwd_noalloc
    fn.argtypes = [P, P, P, P, I64, I64, P, P, P]
    lib.jetfp8_rmsnorm_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.jetfp8_rmsnorm_bwd_workspace_bytes.argtypes = [I64, I64]
    # rows up to 4096 wide never need more than 152 rows of at most 4096 floats
    assert lib.jetfp8_rmsnorm_bwd_workspace_bytes(1 << 24, 4096) == 152 * 4096 * 4
    H = 16384
    # 128 chunks of 128 rows × 16384 columns × 4 B is exactly 8 MiB; one more row is too many
    assert lib.jetfp8_rmsnorm_bwd_workspace_bytes(128 * 128, H) == (8 << 20)
    assert lib.jetfp8_rmsnorm_bwd_workspace_bytes(128 * 128 + 1, H) > (8 << 20)
    A = P(1 << 20)
    assert fn(A, A, A, A, 128 * 128 + 1, H, A, A, None) == 2      # JETFP8_ERR_UNSUPPORTED_SHAPE
    # the largest size passes the size check and stops at the device check (no GPU here)
    assert fn(A, A, A, A, 128 * 128, H, A, A, None) == 4          # JETFP8_ERR_CUDA


def test_rmsnorm_bwd_many_row_chunks_validated(lib):
    """A shape with many rows at a narrow width (more than 65535 128-row chunks,
    the grid's y limit of the wide-row path) is accepted by validation.  Here
    validation stops at the device check (no GPU)."""
    if __import__("torch").cuda.is_available():
        pytest.skip("placeholder addresses: only where no GPU can be reached")
    P, I64, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    fn = lib.jetfp8_rmsnorm_bwd
    fn.argtypes = [P, P, P, P, I64, I64, P, P, P, SZ, P]
    M, H = 128 * 70000, 128
    ws = lib.jetfp8_rmsnorm_bwd_workspace_bytes(M, H)
    A = P(1 << 20)
    assert fn(A, A, A, A, M, H, A, A, A, SZ(ws), None) == 4         # JETFP8_ERR_CUDA, not a shape error


def test_nvfp4_validation(lib):
    """The FP4 entry points check shapes and pointers before the device; the
    block-scale size follows the blocked layout (512-byte atoms of 128 rows ×
    64 elements)."""
    P, I64, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    lib.jetfp8_nvfp4_scale_bytes.restype = SZ
    lib.jetfp8_nvfp4_scale_bytes.argtypes = [I64, I64]
    assert lib.jetfp8_nvfp4_scale_bytes(1, 64) == 512
    assert lib.jetfp8_nvfp4_scale_bytes(128, 4096) == 64 * 512
    assert lib.jetfp8_nvfp4_scale_bytes(129, 4096) == 2 * 64 * 512
    assert lib.jetfp8_nvfp4_scale_bytes(128, 100) == 0
    q = lib.jetfp8_quant_nvfp4
    q.argtypes = [P, I64, I64, P, P, P, P]
    assert q(None, 4, 64, P(64), P(64), P(64), None) == 1            # null input
    assert q(P(64), 0, 64, P(64), P(64), P(64), None) == 1           # R <= 0
    assert q(P(64), 4, 96, P(64), P(64), P(64), None) == 2           # K not a multiple of 64
    assert q(P(48), 4, 64, P(64), P(64), P(64), None) == 3           # bf16 input needs 32 B
    gm = lib.jetfp8_gemm_fprop_nvfp4
    gm.argtypes = [P, P, P, P, P, P, I64, I64, I64, P, P]
    A = P(64)
    assert gm(A, A, A, A, A, A, 4, 384, 256, A, None) == 2           # N not a multiple of 256
    assert gm(A, A, A, A, A, A, 4, 256, 320, A, None) == 2           # K not a multiple of 256
    assert gm(A, A, A, A, A, A, 0, 256, 256, A, None) == 1           # M <= 0
    assert gm(A, None, A, A, A, A, 4, 256, 256, A, None) == 1        # null block scales


def test_grouped_wgrad_validation(lib):
    """The grouped WGrad refuses a bad problem count, null arrays and any
    problem's bad shape or alignment before touching the device."""
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    fn = lib.jetfp8_gemm_wgrad_grouped
    fn.argtypes = [ctypes.c_int, P, P, P, P, I64, P, P, P, ctypes.c_int, P]

    def call(count, M, Ns, Ks, ptr=64, out_dtype=0, arrays=True):
        n = max(len(Ns), 1)
        arr = (P * n)(*([ptr] * n))
        if not arrays:
            return fn(count, None, arr, arr, arr, M, (I64 * n)(*Ns), (I64 * n)(*Ks), arr, out_dtype, None)
        return fn(count, arr, arr, arr, arr, M, (I64 * n)(*Ns), (I64 * n)(*Ks), arr, out_dtype, None)

    assert call(0, 128, [128], [128]) == 1                                 # no problems
    assert call(5, 128, [128] * 5, [128] * 5) == 1                         # above the group limit
    assert call(2, 128, [128, 128], [128, 128], arrays=False) == 1         # null array
    assert call(2, 128, [128, 128], [128, 128], out_dtype=7) == 1          # bad output type
    assert call(2, 100, [128, 128], [128, 128]) == 2                       # M not a multiple of 128
    assert call(3, 256, [128, 384, 200], [128, 128, 128]) == 2             # problem 2's N
    assert call(2, 256, [128, 128], [128, 128], ptr=72) == 3               # misaligned pointers


def test_grouped_quant_weight_validation(lib):
    """The grouped weight quantiser refuses a bad problem count, null arrays and
    any problem's bad shape or alignment before touching the device."""
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    fn = lib.jetfp8_quant_weight_grouped
    fn.argtypes = [ctypes.c_int, P, P, P, P, P, P, P]

    def call(count, Ns, Ks, ptr=64, w=True, q=True, qT=True):
        n = max(len(Ns), 1)
        arr = (P * n)(*([ptr] * n))
        return fn(count, arr if w else None, (I64 * n)(*Ns), (I64 * n)(*Ks), arr if q else None, arr,
                  arr if qT else None, None)

    assert call(0, [128], [128]) == 1                                # no problems
    assert call(5, [128] * 5, [128] * 5) == 1                        # above the group limit
    assert call(2, [128, 128], [128, 128], w=False) == 1             # null weight array
    assert call(2, [128, 128], [128, 128], q=False) == 1             # null code array
    assert call(3, [128, 384, 200], [128, 128, 128]) == 2            # problem 2's N
    assert call(2, [128, 128], [128, 100], qT=False) == 2            # problem 1's K, no transposes
    assert call(2, [128, 128], [128, 128], ptr=72) == 3              # misaligned pointers


def test_failure_hook_validation(lib):
    """The failure-path test hook checks its block index before the device."""
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    fn = lib.jetfp8_test_gemm_fprop_drop_block
    fn.argtypes = [P, P, P, P, I64, I64, I64, P, ctypes.c_int, P]
    assert fn(P(64), P(64), P(64), P(64), 4, 128, 256, P(64), 2, None) == 1    # K/128 = 2 blocks
    assert fn(P(64), P(64), P(64), P(64), 4, 128, 256, P(64), -1, None) == 1
    assert fn(P(64), P(64), P(64), P(64), 4, 128, 200, P(64), 0, None) == 2    # K not a multiple of 128


def test_launch_logging(tmp_path):
    """JETFP8_LOG=1 makes every entry point print its name and sizes to stderr
    (before its arguments are checked, so no GPU is needed); unset, nothing."""
    import subprocess
    import sys
    code = ("import ctypes\n"
            "from fp8_mixed_granularity_gb300 import jetfp8 as J\n"
            "lib = J.load_library()\n"
            "P = ctypes.c_void_p\n"
            "assert lib.jetfp8_quant_act_1x128(P(64), 4, 100, P(64), P(64), None) == 2\n")
    env = dict(os.environ, PYTHONPATH=ROOT)
    env.pop("JETFP8_LOG", None)
    quiet = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True)
    assert quiet.returncode == 0, quiet.stderr
    assert "jetfp8:" not in quiet.stderr
    env["JETFP8_LOG"] = "1"
    loud = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True)
    assert loud.returncode == 0, loud.stderr
    assert "jetfp8: jetfp8_quant_act_1x128 4 100" in loud.stderr


def test_no_cpu_fallback(lib, tmp_path):
    """The binding refuses host tensors (there is no CPU path), and without the
    built library the first call raises instead of computing anything."""
    import subprocess
    import sys
    import torch
    from fp8_mixed_granularity_gb300 import jetfp8 as J
    x = torch.zeros(4, 128, dtype=torch.bfloat16)
    q = torch.zeros(4, 128, dtype=torch.uint8)
    s = torch.zeros(1, 4, dtype=torch.float32)
    with pytest.raises(J.JetFP8Error, match="CUDA tensor"):
        J.jetfp8_quant_act_1x128(x, q, s)
    code = ("from fp8_mixed_granularity_gb300 import jetfp8 as J\n"
            f"J.LIB_PATH = {str(tmp_path / 'missing.so')!r}\n"
            "try:\n"
            "    J.load_library(J.LIB_PATH)\n"
            "except J.JetFP8Error as e:\n"
            "    print('raised:', e)\n")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=dict(os.environ, PYTHONPATH=ROOT),
                         capture_output=True, text=True)
    assert out.returncode == 0 and "raised:" in out.stdout and "not found" in out.stdout
