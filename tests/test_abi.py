"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, and rejects bad arguments on the host before touching CUDA.

The pointer values used here are never dereferenced: every call below returns
from the host-side checks (or the empty-problem shortcut) before any launch.
"""
import ctypes
import os
import re
import subprocess

import pytest

import selective_state_space_132_b300 as ssm
from selective_state_space_132_b300 import binding as bd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssm.h")

OK, INVALID, UNSUPPORTED, ALIGN, WORKSPACE = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    ssm.build_library()
    return ssm.load_library()


def header_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SSM_API\s+[\w\s\*]+?\b(ssm_\w+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    fns = header_functions()
    for name in ("ssm_scan_fwd", "ssm_ssd_chunk_fwd", "ssm_step_decode", "ssm_ssd_plan",
                 "ssm_scan_workspace_size", "ssm_ssd_workspace_size", "ssm_status_string",
                 "ssm_version", "ssm_read_device_status", "ssm_conv1d", "ssm_scan_bwd",
                 "ssm_scan_bwd_workspace_size"):
        assert name in fns


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", ssm.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)$", out, flags=re.M))
    for name in header_functions():
        assert name in exported, name
        assert hasattr(lib, name)
    # nothing but the C ABI is exported
    assert all(n.startswith("ssm_") or n.startswith("_") for n in exported), exported


def test_version_and_status_strings(lib):
    assert ssm.version() >= 10000
    for code in range(7):
        assert lib.ssm_status_string(code)
    assert lib.ssm_status_string(99) == b"unknown status"


def _scan(**kw):
    base = dict(batch=2, seqlen=64, dim=32, dstate=16, time_chunk=0, io_dtype=1,
                delta_softplus=1, x=0x10000, delta=0x20000, B=0x30000, C=0x40000, z=None,
                A=0x50000, D=None, delta_bias=None, h0=None, y=0x60000, h_final=None,
                workspace=None, workspace_bytes=0)
    base.update(kw)
    return bd.ScanArgs(**base)


def _scan_rc(lib, **kw):
    a = _scan(**kw)
    return lib.ssm_scan_fwd(ctypes.byref(a), None)


def test_scan_rejects_bad_arguments(lib):
    assert lib.ssm_scan_fwd(None, None) == INVALID
    assert _scan_rc(lib, dstate=0) == INVALID
    assert _scan_rc(lib, batch=-1) == INVALID
    assert _scan_rc(lib, io_dtype=7) == INVALID
    assert _scan_rc(lib, delta_softplus=2) == INVALID
    assert _scan_rc(lib, time_chunk=33) == INVALID
    a = _scan()
    a.discretization = 2                               # neither Euler nor ZOH
    assert lib.ssm_scan_fwd(ctypes.byref(a), None) == INVALID
    assert _scan_rc(lib, dstate=65) == UNSUPPORTED
    assert _scan_rc(lib, batch=70000) == UNSUPPORTED
    assert _scan_rc(lib, x=None) == INVALID
    assert _scan_rc(lib, A=None) == INVALID
    assert _scan_rc(lib, x=0x10001) == ALIGN            # bf16 needs 2-byte alignment
    assert _scan_rc(lib, A=0x50002) == ALIGN            # fp32 needs 4-byte alignment
    assert _scan_rc(lib, io_dtype=0, x=0x10002) == ALIGN
    assert _scan_rc(lib, y=0x10000) == INVALID          # y aliases x
    assert _scan_rc(lib, y=0x30010) == INVALID          # y overlaps B
    # a forced time split needs a workspace
    assert _scan_rc(lib, time_chunk=32) == WORKSPACE
    need = ctypes.c_size_t(0)
    a = _scan(time_chunk=32)
    assert lib.ssm_scan_workspace_size(ctypes.byref(a), ctypes.byref(need)) == OK
    assert need.value > 0
    assert _scan_rc(lib, time_chunk=32, workspace=0x70000, workspace_bytes=need.value - 1) \
        == WORKSPACE
    assert _scan_rc(lib, time_chunk=32, workspace=0x70010, workspace_bytes=need.value) == ALIGN


def test_scan_plan(lib):
    assert ssm.scan_plan(8, 2048, 1536, 16) == (2048, 1, 1)          # one pass, no split
    cl, k, n = ssm.scan_plan(1, 131072, 2048, 16)                   # long: split over time,
    assert k > 1 and n == 1 and cl % 32 == 0 and cl * k >= 131072   # one launch (look-back)
    assert ssm.scan_plan(2, 300, 8, 16, time_chunk=64) == (64, 5, 1)
    # shapes the TMA kernel does not take run the summary pass as a launch of its own
    assert ssm.scan_plan(2, 300, 7, 16, time_chunk=64) == (64, 5, 2)
    assert ssm.scan_plan(0, 300, 8, 16)[2] == 0


def test_scan_workspace_holds_status_word_and_chunk_summaries(lib):
    # one time chunk: only the 256-byte device status word
    assert ssm.scan_workspace_size(8, 2048, 1536, 16) == 256
    # the long-context shape is split over time: status word + per-chunk end states
    cl, k, launches = ssm.scan_plan(1, 131072, 2048, 16)
    assert k > 1 and launches == 1
    # status word, end states (B, K, D, N), step sums (B, K, D), ticket + one flag per
    # (batch row, chunk, 32-channel slab)
    need = (256 + (1 * k * 2048 * 16 * 4 + 255) // 256 * 256 + (k * 2048 * 4 + 255) // 256 * 256
            + ((1 + k * (2048 // 32)) * 4 + 255) // 256 * 256)
    assert ssm.scan_workspace_size(1, 131072, 2048, 16) == need


def test_empty_problems_return_without_launch(lib):
    assert _scan_rc(lib, batch=0) == OK
    assert _scan_rc(lib, dim=0, A=None) == OK


def _ssd(**kw):
    base = dict(batch=1, seqlen=64, nheads=4, headdim=64, ngroups=1, dstate=64, chunk_size=0,
                io_dtype=1, delta_softplus=1, x=0x100000, delta=0x200000, B=0x300000,
                C=0x400000, z=None, A=0x500000, D=None, delta_bias=None, h0=None,
                y=0x600000, h_final=None, workspace=None, workspace_bytes=0)
    base.update(kw)
    return bd.SSDArgs(**base)


def test_ssd_rejects_bad_arguments(lib):
    def rc(**kw):
        a = _ssd(**kw)
        return lib.ssm_ssd_chunk_fwd(ctypes.byref(a), None)
    assert rc(ngroups=3) == INVALID
    assert rc(nheads=0) == INVALID
    assert rc(dstate=257) == UNSUPPORTED
    assert rc(A=None) == INVALID
    assert rc(B=0x300001) == ALIGN
    assert rc(y=0x100000) == INVALID
    assert rc() == WORKSPACE
    need = ctypes.c_size_t(0)
    a = _ssd()
    assert lib.ssm_ssd_workspace_size(ctypes.byref(a), ctypes.byref(need)) == OK
    assert need.value >= 256
    assert rc(workspace=0x700080, workspace_bytes=need.value) == ALIGN
    assert rc(batch=0, workspace=0x700000, workspace_bytes=need.value) == OK


def test_noalloc_scan_rejects_problems_beyond_its_scratch(lib):
    """Sizes whose chunk summaries exceed the fixed 4 MiB buffer are refused on the
    host, before any CUDA call (so this runs without a GPU)."""
    from conftest import cuda_available
    if cuda_available():
        pytest.skip("uses fake device pointers; checked on CPU-only hosts")
    # 64 chunks x 1024 channels x (16 + 1) floats > 4 MiB
    far = dict(x=1 << 32, delta=2 << 32, B=3 << 32, C=4 << 32, A=5 << 32, y=6 << 32)
    a = _scan(batch=1, seqlen=2048, dim=1024, time_chunk=32, **far)
    need = ctypes.c_size_t(0)
    assert lib.ssm_scan_workspace_size(ctypes.byref(a), ctypes.byref(need)) == OK
    assert need.value > bd.NOALLOC_SCRATCH_BYTES
    assert lib.ssm_scan_fwd_noalloc(ctypes.byref(a), None) == UNSUPPORTED
    assert lib.ssm_scan_fwd_noalloc(None, None) == INVALID
    assert lib.ssm_scan_fwd_noalloc(ctypes.byref(_scan(x=0x10001)), None) == ALIGN
    assert lib.ssm_scan_fwd_noalloc(ctypes.byref(_scan(batch=0)), None) == OK


def test_decode_rejects_bad_arguments(lib):
    def rc(**kw):
        base = dict(batch=4, dim=32, dstate=16, io_dtype=1, delta_softplus=1, state=0x100000,
                    x=0x200000, delta=0x300000, B=0x400000, C=0x500000, z=None, A=0x600000,
                    D=None, delta_bias=None, y=0x700000)
        base.update(kw)
        a = bd.DecodeArgs(**base)
        return lib.ssm_step_decode(ctypes.byref(a), None)
    assert rc(state=None) == INVALID
    assert rc(dstate=0) == INVALID
    assert rc(dstate=65) == UNSUPPORTED
    assert rc(state=0x100002) == ALIGN
    assert rc(y=0x200000) == INVALID
    assert rc(y=0x100000) == INVALID                    # y inside the state
    assert rc(batch=0) == OK


def test_ssd_decode_rejects_bad_arguments(lib):
    def rc(**kw):
        base = dict(batch=2, nheads=4, headdim=64, ngroups=1, dstate=128, io_dtype=1,
                    delta_softplus=1, state=0x100000, x=0x200000, delta=0x300000, B=0x400000,
                    C=0x500000, z=None, A=0x600000, D=None, delta_bias=None, y=0x700000)
        base.update(kw)
        a = bd.SSDDecodeArgs(**base)
        return lib.ssm_ssd_step_decode(ctypes.byref(a), None)
    assert lib.ssm_ssd_step_decode(None, None) == INVALID
    assert rc(ngroups=3) == INVALID                  # H % G != 0
    assert rc(dstate=300) == UNSUPPORTED
    assert rc(state=None) == INVALID
    assert rc(x=0x200001) == ALIGN
    assert rc(y=0x200000) == INVALID                 # y aliases x
    assert rc(batch=0) == OK                         # nothing to do, nothing launched


def test_scan_bwd_rejects_bad_arguments(lib):
    def args(**kw):
        base = dict(batch=2, seqlen=64, dim=32, dstate=16, io_dtype=1, delta_softplus=1,
                    discretization=0, reserved=0, x=0x100000, delta=0x200000, B=0x300000,
                    C=0x400000, z=None, A=0x500000, D=None, delta_bias=None, h0=None,
                    dy=0x600000, dh_final=None, dx=0x700000, ddelta=0x800000, dz=None,
                    dA=0x900000, dB=0xa00000, dC=0xb00000, dD=None, ddelta_bias=None,
                    dh0=None, workspace=None, workspace_bytes=0)
        base.update(kw)
        return bd.ScanBwdArgs(**base)

    def rc(**kw):
        a = args(**kw)
        return lib.ssm_scan_bwd(ctypes.byref(a), None)
    assert lib.ssm_scan_bwd(None, None) == INVALID
    assert rc(dstate=0) == INVALID
    assert rc(dstate=65) == UNSUPPORTED
    assert rc(discretization=3) == INVALID
    assert rc(dy=None) == INVALID
    assert rc(dB=None) == INVALID
    assert rc(z=0xc00000) == INVALID                 # z without dz
    assert rc(dz=0xc00000) == INVALID                # dz without z
    assert rc(dx=0x100001) == ALIGN
    assert rc(dA=0x900002) == ALIGN
    assert rc(dx=0x100000) == INVALID                # dx aliases x
    assert rc(ddelta=0x700010) == INVALID            # two outputs overlap
    assert rc(dB=0x200000) == INVALID                # output over an input
    need = ctypes.c_size_t(0)
    a = args()
    assert lib.ssm_scan_bwd_workspace_size(ctypes.byref(a), ctypes.byref(need)) == OK
    # status word + one state per (b, 16-step tile, d): 2 * 4 * 32 * 16 floats
    assert need.value == 256 + 2 * 4 * 32 * 16 * 4
    assert ssm.scan_bwd_workspace_size(8, 2048, 1536, 16) == 256 + 8 * 128 * 1536 * 16 * 4


def test_conv1d_rejects_bad_arguments(lib):
    def rc(**kw):
        base = dict(batch=2, seqlen=64, dim=32, width=4, io_dtype=1, silu=1, x=0x100000,
                    x_prev=None, weight=0x200000, bias=None, out=0x300000)
        base.update(kw)
        a = bd.Conv1dArgs(**base)
        return lib.ssm_conv1d(ctypes.byref(a), None)
    assert lib.ssm_conv1d(None, None) == INVALID
    assert rc(width=0) == INVALID
    assert rc(width=9) == UNSUPPORTED
    assert rc(silu=2) == INVALID
    assert rc(io_dtype=5) == INVALID
    assert rc(weight=None) == INVALID
    assert rc(x=0x100001) == ALIGN
    assert rc(weight=0x200002) == ALIGN
    assert rc(out=0x100000) == INVALID               # out aliases x
    assert rc(out=0x400000, x_prev=0x400010) == INVALID   # out overlaps x_prev
    assert rc(workspace=0xc00000, workspace_bytes=128) == WORKSPACE   # status word is 256 B
    assert rc(workspace=0xc00010, workspace_bytes=256) == ALIGN
    assert rc(seqlen=0) == OK                        # nothing to do, nothing launched


def test_ops_fail_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(bd, "_lib", None)
    monkeypatch.setattr(bd, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        bd.load_library()


def test_header_is_plain_c_and_callable_from_c(lib, tmp_path):
    """A C99 program compiles against include/ssm.h with -Werror -pedantic, links
    against the library and runs its host-only entry points."""
    import shutil
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "probe"
    libdir = os.path.dirname(ssm.library_path())
    src = os.path.join(ROOT, "tests", "c_abi_probe.c")
    build = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                            "-I", os.path.join(ROOT, "include"), src, "-o", str(exe),
                            "-L", libdir, "-l:" + os.path.basename(ssm.library_path()),
                            "-Wl,-rpath," + libdir], capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "0 failure(s)" in run.stdout
