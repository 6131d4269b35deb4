"""Host-side checks of the C ABI that need no GPU: the library builds and loads,
exports every symbol include/fa_attention.h declares, and rejects bad arguments
before touching any device."""
import ctypes
import os
import re

import pytest

from exact_attention_37_gb300 import _lib
from exact_attention_37_gb300 import build as fabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa_attention.h")


@pytest.fixture(scope="module")
def lib():
    fabuild.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    return sorted({n for n in names if n.startswith("fa_")})


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_check_device_status", "fa_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_device_check_selftest_needs_the_checked_build(lib):
    # the release library has the device-side checks compiled out
    assert lib.fa_selftest_device_check(1, None) == 2


def test_status_strings(lib):
    for code, name in _lib.STATUS.items():
        assert lib.fa_status_string(code).decode() == name
    assert lib.fa_version() >> 16 == 1


def fwd(lib, **over):
    a = dict(q=16, k=16, v=16, o=16, lse=16, B=1, H=1, N=8, d=64, scale=0.125, causal=0, dtype=1)
    a.update(over)
    vp = ctypes.c_void_p
    return lib.fa_fwd(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["o"]), vp(a["lse"]), a["B"], a["H"], a["N"], a["d"],
                      a["scale"], a["causal"], a["dtype"], None)


@pytest.mark.parametrize("over,code", [
    (dict(d=96), 2), (dict(d=32), 2), (dict(d=512), 2),
    (dict(N=-1), 1), (dict(B=-2), 1), (dict(H=-1), 1),
    (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1), (dict(scale=0.0), 1), (dict(scale=-1.0), 1),
    (dict(dtype=7), 1),
    (dict(q=0), 1), (dict(lse=0), 1),
    (dict(k=24), 3), (dict(o=8), 3),
])
def test_fwd_rejects_bad_arguments_on_the_host(lib, over, code):
    assert fwd(lib, **over) == code


def test_grouped_and_unequal_lengths_validation(lib):
    vp = ctypes.c_void_p
    p = [vp(16)] * 5

    def ex(B=1, H=4, Hkv=2, Nq=8, Nk=8, d=64):
        return lib.fa_fwd_ex(*p, B, H, Hkv, Nq, Nk, d, 0.125, 1, 1, None)

    assert ex(Hkv=3) == 1      # H_kv must divide H
    assert ex(Hkv=0) == 1
    assert ex(Nk=-1) == 1
    assert ex(Nk=0) == 2       # queries with an empty key set
    assert ex(Nq=0) == 0       # no query rows: nothing to do
    assert ex(d=80) == 2


def test_fwd_empty_problem_is_a_no_op(lib):
    assert fwd(lib, N=0, q=0, k=0, v=0, o=0, lse=0) == 0
    assert fwd(lib, B=0) == 0


def bwd(lib, ws_bytes=None, **over):
    a = dict(p=256, ws=256, B=1, H=2, N=10, d=128, scale=0.1, causal=1, dtype=0)
    a.update(over)
    vp = ctypes.c_void_p
    ws_bytes = lib.fa_bwd_workspace_size(a["B"], a["H"], a["N"], a["d"]) if ws_bytes is None else ws_bytes
    ptrs = [vp(a.get(n, a["p"])) for n in ("q", "k", "v", "o", "do", "lse", "dq", "dk", "dv")]
    return lib.fa_bwd(*ptrs, vp(a["ws"]), ws_bytes, a["B"], a["H"], a["N"], a["d"], a["scale"], a["causal"],
                      a["dtype"], None)


def test_bwd_rejects_bad_arguments_on_the_host(lib):
    assert bwd(lib, d=80) == 2
    assert bwd(lib, dq=0) == 1
    assert bwd(lib, dk=40) == 3
    assert bwd(lib, ws=0) == 4
    assert bwd(lib, ws_bytes=100) == 4
    assert bwd(lib, ws=256 + 16) == 3  # workspace must be 256-byte aligned
    assert bwd(lib, B=0) == 0


def test_noalloc_backward_rejects_oversized_problems_on_the_host(lib):
    vp = ctypes.c_void_p
    args = [vp(256)] * 9
    # The fixed scratch holds 32 MiB and the workspace is 8 bytes per (padded) row at
    # every head dimension: 4,194,304 rows fit exactly, one more does not.
    for d in (64, 128, 256):
        assert lib.fa_bwd_workspace_size(1, 1, 4194304, d) == 33554432
        assert lib.fa_bwd_workspace_size(1, 1, 4194304 + 1, d) > 33554432
        assert lib.fa_bwd_noalloc(*args, 1, 1, 4194304 + 1, d, 0.1, 0, 1, None) == 4
        assert lib.fa_bwd_noalloc(*args, 2, 2, 1048577, d, 0.1, 0, 1, None) == 4
    assert lib.fa_bwd_noalloc(*args, 1, 1, 8, 96, 0.1, 0, 1, None) == 2
    assert lib.fa_bwd_noalloc(*args, 0, 1, 8, 64, 0.1, 0, 1, None) == 0


def test_workspace_is_linear_in_n(lib):
    for d in (64, 128, 256):
        # L log2 e and D, fp32, for every row: no kernel keeps a gradient accumulator
        sizes = [lib.fa_bwd_workspace_size(2, 16, n, d) for n in (1024, 2048, 4096, 8192)]
        for n, s in zip((1024, 2048, 4096, 8192), sizes):
            assert s == 2 * 16 * n * 2 * 4
    # L and D rows are padded per head to a multiple of 128, each part 256-byte aligned
    for d in (64, 128, 256):
        assert lib.fa_bwd_workspace_size(1, 1, 1, d) == 2 * 512
        assert lib.fa_bwd_workspace_size(3, 1, 129, d) == 2 * 3 * 256 * 4
    assert lib.fa_bwd_workspace_size(1, 1, 0, 64) == 0
    assert lib.fa_bwd_workspace_size(1, 1, 8, 96) == 0


def test_valid_call_without_a_device_reports_cuda_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert fwd(lib) in (2, 5)


def test_selftest_rejects_bad_limits_on_the_host(lib):
    # validated before any device work: 0 < limit_us <= 1 s
    assert lib.fa_selftest_wait_timeout(0, None) == 1
    assert lib.fa_selftest_wait_timeout(1000001, None) == 1


def test_host_entry_points_validate_on_the_host(lib):
    vp = ctypes.c_void_p
    assert lib.fa_host_scratch_size(2, 3, 100, 128, 1) > lib.fa_host_scratch_size(2, 3, 100, 128, 0) > 0
    assert lib.fa_host_scratch_size(1, 1, 8, 96, 1) == 0
    assert lib.fa_host_scratch_size(0, 1, 8, 64, 1) == 0
    p = vp(4096)
    # empty problem: nothing to do
    assert lib.fa_fwd_bwd_host(*([p] * 9), p, 1 << 20, 0, 2, 64, 64, 0.1, 0, 1, 0, None) == 0
    # null input, missing scratch, small scratch, misaligned scratch: refused before any device work
    assert lib.fa_fwd_bwd_host(*([vp(0)] + [p] * 8), p, 1 << 30, 1, 2, 64, 64, 0.1, 0, 1, 0, None) == 1
    assert lib.fa_fwd_bwd_host(*([p] * 9), vp(0), 1 << 30, 1, 2, 64, 64, 0.1, 0, 1, 0, None) == 4
    assert lib.fa_fwd_bwd_host(*([p] * 9), p, 100, 1, 2, 64, 64, 0.1, 0, 1, 0, None) == 4
    assert lib.fa_fwd_host(*([p] * 5), vp(4096 + 16), 1 << 30, 1, 2, 64, 64, 0.1, 0, 1, 0, None) == 3


@pytest.mark.parametrize("B,H,N,chunks", [(2, 16, 8192, 0), (4, 16, 2048, 0), (1, 1, 256, 0), (2, 3, 777, 0),
                                          (1, 5, 513, 0), (2, 8, 256, 0), (2, 16, 8192, 4), (2, 16, 8192, 3),
                                          (2, 16, 8192, 64), (1, 100, 1000, 64), (5, 7, 33, 0), (8, 125, 64, 0)])
def test_host_chunk_plan_covers_every_head_once(lib, B, H, N, chunks):
    plan = _lib.fa_host_chunk_plan(B, H, N, chunks)
    BH = B * H
    assert sum(plan) == BH and all(c > 0 for c in plan) and 1 <= len(plan) <= 64
    # every chunk start keeps L (B*H rows of N floats) 16-byte aligned
    starts = [sum(plan[:i]) for i in range(len(plan))]
    assert all(s * N % 4 == 0 for s in starts)
    if chunks > 0:  # an explicit count: equal chunks, the last one possibly smaller
        assert len(plan) <= max(chunks, 1) or len(plan) <= 64
        assert all(c == plan[0] for c in plan[:-1]) and plan[-1] <= plan[0]


def test_host_chunk_plan_default_is_tapered(lib):
    assert _lib.fa_host_chunk_plan(2, 16, 8192) == [4, 8, 8, 8, 4]
    assert _lib.fa_host_chunk_plan(4, 16, 2048) == [8, 16, 16, 16, 8]
    assert _lib.fa_host_chunk_plan(2, 16, 8192, 4) == [8, 8, 8, 8]
    assert _lib.fa_host_chunk_plan(1, 1, 256) == [1]
    assert lib.fa_host_chunk_plan(0, 4, 128, 0, None, 0) == 0
    assert lib.fa_host_chunk_plan(-1, 4, 128, 0, None, 0) == -1


@pytest.mark.parametrize("nheads", [1, 2, 7, 32, 64, 96, 1000])
@pytest.mark.parametrize("nblocks", [1, 16, 64, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_cta_head_group_properties(lib, nheads, nblocks, causal):
    sms, bph = 152, 8 << 20
    g = _lib.fa_cta_head_group(nheads, nblocks, bph, causal, sms)
    assert 1 <= g <= nheads
    work = nblocks * (nblocks + 1) // 2 if causal else nblocks * nblocks
    g_tail = -(-sms * nblocks // work)
    g_l2 = max(1, (48 << 20) // bph)
    g0 = min(max(g_tail, g_l2), nheads)
    assert g >= g0  # no tail inside a group, and about 48 MB of tensors per group
    divisors = [c for c in range(g0, min(2 * g0, nheads) + 1) if nheads % c == 0]
    assert g == (divisors[0] if divisors else g0)  # equal groups whenever a divisor is near


def test_cta_head_group_at_the_workload_shapes(lib):
    # long workload (32 heads, 8 MB of Q, K, V, O or dO per head), 152 SMs
    assert _lib.fa_cta_head_group(32, 32, 8 << 20, True, 152) == 16   # forward: 256-row blocks
    assert _lib.fa_cta_head_group(32, 64, 8 << 20, True, 152) == 8    # backward: 128-row blocks
    assert _lib.fa_cta_head_group(32, 256, 32 << 20, True, 152) == 2  # 32k context, backward
    assert _lib.fa_cta_head_group(64, 16, 1 << 20, False, 152) == 64  # small heads: one group
    assert lib.fa_cta_head_group(0, 4, 1, 0, 152) == -1


def test_nvtx_ranges_compile(tmp_path):
    """The optional NVTX build (-DFA_NVTX: a range around every C-ABI call) compiles."""
    import subprocess

    for src in ("fa_api.cu", "fa_host.cu"):
        cmd = [fabuild.nvcc(), *fabuild.ARCH, *fabuild.FLAGS, "-DFA_NVTX", "-c", os.path.join(fabuild.CSRC, src),
               "-o", str(tmp_path / (src + ".o"))]
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
