"""The C-ABI library builds for sm_103a, loads, exports every function the
public header declares, and rejects bad arguments on the host before touching
a GPU (these checks return before any CUDA call, so they run without one)."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

import combine_moe_layout_05_gb300 as moe
from combine_moe_layout_05_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.load()


def test_header_declares_the_boundary():
    names = moe.declared_functions()
    for n in ["moe_layout", "moe_dispatch", "moe_combine",
              "moe_layout_workspace_bytes", "moe_status_string"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            for name in moe.declared_functions(os.path.join(ROOT, "include", h)):
                assert hasattr(lib, name), name


def test_status_strings(lib):
    assert moe.moe_status_string(0) == "ok"
    assert "alignment" in moe.moe_status_string(2) or "misaligned" in moe.moe_status_string(2)
    assert moe.moe_status_string(99) == "unknown status"


def test_workspace_query(lib):
    assert moe.moe_layout_workspace_bytes(128, 8, 256) == 0          # one block
    ws = moe.moe_layout_workspace_bytes(16384, 8, 128)
    assert ws > 0 and ws % 256 == 0
    assert moe.moe_layout_workspace_bytes(16384, 8, 100000) == 0     # invalid E


# Fake, never-dereferenced device addresses: the host checks reject the call
# before anything is launched.
FAKE = 0x10000
P = ctypes.c_void_p


def _layout(lib, ids=FAKE, T=4, K=2, E=8, R=2, outs=FAKE, ws=None, wsb=0):
    return lib.moe_layout(P(ids), T, K, E, R, P(outs), P(outs), P(outs),
                          P(outs), P(outs), None, P(ws) if ws else None, wsb, None)


def test_layout_host_checks(lib):
    assert _layout(lib, E=8, R=3) == 1            # E % R != 0
    assert _layout(lib, K=9, E=8) == 1            # K > E
    assert _layout(lib, K=33, E=64) == 1          # K > MOE_MAX_TOPK
    assert _layout(lib, E=2048, R=2) == 1         # E > MOE_MAX_EXPERTS
    assert _layout(lib, T=-1) == 1
    assert _layout(lib, ids=0) == 1               # null ids with T > 0
    assert _layout(lib, outs=0) == 1
    assert _layout(lib, ids=FAKE + 2) == 2        # misaligned
    assert _layout(lib, T=100000, K=8, E=128, R=16) == 4   # workspace missing
    need = moe.moe_layout_workspace_bytes(100000, 8, 128)
    assert _layout(lib, T=100000, K=8, E=128, R=16, ws=FAKE, wsb=need - 1) == 4
    assert _layout(lib, T=100000, K=8, E=128, R=16, ws=FAKE + 8, wsb=need) == 2
    assert _layout(lib, T=2**28, K=16, E=64, R=1) == 1     # T*K >= 2^31


def test_dispatch_host_checks(lib):
    d = lib.moe_dispatch
    assert d(P(FAKE), 4, 100, 2, P(FAKE), 0, P(FAKE), None, None) == 1   # H % 8
    assert d(P(FAKE), 4, 136, 2, P(FAKE), 1, P(FAKE), P(FAKE), None) == 1  # H % 128 (fp8)
    assert d(P(FAKE), 4, 128, 2, P(FAKE), 1, P(FAKE), None, None) == 1   # no scales
    assert d(P(FAKE), 4, 128, 2, P(FAKE), 2, P(FAKE), None, None) == 1   # bad fp8 flag
    assert d(P(FAKE + 8), 4, 128, 2, P(FAKE), 0, P(FAKE), None, None) == 2
    assert d(P(FAKE), 4, 128, 2, P(FAKE), 0, P(FAKE + 4), None, None) == 2
    assert d(None, 4, 128, 2, P(FAKE), 0, P(FAKE), None, None) == 1
    assert d(None, 0, 128, 2, None, 0, None, None, None) == 0          # T == 0: no-op


def test_combine_host_checks(lib):
    c = lib.moe_combine
    assert c(P(FAKE), P(FAKE), P(FAKE), 4, 12, 2, P(FAKE), None) == 1    # H % 8
    assert c(P(FAKE), P(FAKE), P(FAKE), 4, 128, 0, P(FAKE), None) == 1   # K == 0
    assert c(P(FAKE + 8), P(FAKE), P(FAKE), 4, 128, 2, P(FAKE), None) == 2
    assert c(P(FAKE), P(FAKE + 2), P(FAKE), 4, 128, 2, P(FAKE), None) == 2
    assert c(P(FAKE), P(FAKE), None, 4, 128, 2, P(FAKE), None) == 1
    assert c(None, None, None, 0, 128, 2, None, None) == 0              # T == 0: no-op


def test_layout_dispatch_plan_query(lib):
    # decode shapes run as one kernel; prefill shapes as the counting kernel
    # plus one rank-and-pack grid; shapes whose ranking blocks would need too
    # much shared memory for the packing blocks' occupancy (E = 1024) as
    # moe_layout's launches and then the dispatch kernel
    assert moe.moe_layout_dispatch_kernels(128, 7168, 8, 256, False) == 1
    assert moe.moe_layout_dispatch_kernels(256, 7168, 8, 256, True) == 1
    assert moe.moe_layout_dispatch_kernels(4096, 7168, 8, 384, False) == 2
    assert moe.moe_layout_dispatch_kernels(16384, 4096, 8, 128, True) == 2
    assert moe.moe_layout_dispatch_kernels(16384, 7168, 8, 256, True) == 2
    assert moe.moe_layout_dispatch_kernels(1000, 4096, 8, 128, False) == 2
    assert moe.moe_layout_dispatch_kernels(5000, 65536, 8, 16, False) == 2
    assert moe.moe_layout_dispatch_kernels(2000, 1024, 8, 1024, False) == 3    # 2 + dispatch
    assert moe.moe_layout_dispatch_kernels(30000, 1024, 8, 1024, False) == 4   # 3 + dispatch
    # moe_layout alone: one self-counting launch, count + ranking blocks
    # (while the ranking blocks' shared memory fits), or count, scan, rank
    assert moe.moe_layout_kernels(128, 8, 256) == 1
    assert moe.moe_layout_kernels(4096, 8, 384) == 2                 # count + ranking
    assert moe.moe_layout_kernels(16384, 8, 128) == 2
    assert moe.moe_layout_kernels(2000, 8, 1024) == 2
    assert moe.moe_layout_kernels(30000, 8, 1024) == 3               # count, scan, rank
    assert moe.moe_layout_kernels(16384, 8, 100000) == 0             # invalid E
    assert moe.moe_layout_dispatch_kernels(512, 7168, 8, 256, False) == 2
    assert moe.moe_layout_dispatch_kernels(0, 128, 4, 16, False) == 1
    assert moe.moe_layout_dispatch_kernels(128, 100, 8, 256, False) == 0    # H % 8
    assert moe.moe_layout_dispatch_kernels(128, 136, 8, 256, True) == 0     # H % 128


def test_layout_dispatch_host_checks(lib):
    f = lib.moe_layout_dispatch
    args = lambda **kw: [P(kw.get("ids", FAKE)), P(kw.get("tok", FAKE)), kw.get("T", 4),
                         kw.get("H", 128), kw.get("K", 2), kw.get("E", 8), kw.get("R", 2),
                         kw.get("fp8", 0), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                         None, P(kw.get("packed", FAKE)), P(kw.get("scales", FAKE)),
                         P(kw.get("ws")) if kw.get("ws") else None, kw.get("wsb", 0), None]
    assert f(*args(E=8, R=3)) == 1
    assert f(*args(H=100)) == 1
    assert f(*args(H=136, fp8=1)) == 1
    assert f(*args(tok=FAKE + 8)) == 2
    assert f(*args(packed=FAKE + 4)) == 2
    assert f(*args(fp8=1, scales=FAKE + 2)) == 2
    assert f(*args(T=4096, H=7168, K=8, E=384, R=48)) == 4       # needs workspace


def test_workspace_fits_the_static_scratch(lib):
    # moe_layout_static's documented bound: every batch moe_layout accepts
    # with E >= 2 needs at most MOE_LAYOUT_STATIC_SCRATCH_BYTES of workspace
    # (both multi-launch forms: count/scan/rank and counting clusters plus
    # ranking blocks); with E = 1 only batches of more than 12.5 M entries
    # need more
    scratch = 96 << 10
    Ts = sorted({int(x) for x in np.geomspace(500, 20_000_000, 60)} | {4097, 16384, 30000})
    for E in (1, 2, 3, 8, 64, 128, 256, 384, 512, 1000, 1024):
        for K in (1, 2, 8, 32):
            if K > E:
                continue
            for T in Ts:
                if moe.moe_layout_kernels(T, K, E) == 0:
                    continue                          # not accepted
                ws = moe.moe_layout_workspace_bytes(T, K, E)
                if E >= 2 or T * K <= 12_500_000:
                    assert ws <= scratch, (T, K, E, ws)


def test_layout_size_limit(lib):
    # the shared-memory bound of the kernels: at least 6.5e8 / E entries
    for E in (128, 384, 1024):
        T = int(6.5e8 / E) // 8
        assert moe.moe_layout_workspace_bytes(T, 8, E) > 0
    assert moe.moe_layout_workspace_bytes(2_000_000, 8, 1024) == 0      # too large
    assert _layout(lib, T=2_000_000, K=8, E=1024, R=1) == 1


def test_combine_fp8_host_checks(lib):
    c = lib.moe_combine_fp8
    args = lambda **kw: [P(kw.get("q", FAKE)), P(kw.get("s", FAKE)), P(FAKE), P(FAKE),
                         kw.get("T", 4), kw.get("H", 256), kw.get("K", 2), P(kw.get("o", FAKE)), None]
    assert c(*args(H=200)) == 1                  # H % 128
    assert c(*args(K=0)) == 1
    assert c(*args(q=FAKE + 8)) == 2
    assert c(*args(s=FAKE + 2)) == 2
    assert c(*args(o=FAKE + 4)) == 2
    assert c(None, None, None, None, 0, 256, 2, None, None) == 0   # T == 0: no-op


def test_combine_rank_partial_host_checks(lib):
    c = lib.moe_combine_rank_partial
    args = lambda **kw: [P(kw.get("y", FAKE)), P(FAKE), P(kw.get("ids", FAKE)), P(FAKE),
                         kw.get("T", 4), kw.get("H", 64), kw.get("K", 2), kw.get("E", 8),
                         kw.get("R", 2), P(kw.get("o", FAKE)), None]
    assert c(*args(R=3)) == 1                    # E % R
    assert c(*args(E=2000, R=1)) == 1            # E > MOE_MAX_EXPERTS
    assert c(*args(H=12)) == 1
    assert c(*args(y=FAKE + 8)) == 2
    assert c(*args(ids=FAKE + 2)) == 2
    assert c(None, None, None, None, 0, 64, 2, 8, 2, None, None) == 0


def test_missing_library_fails_loudly(tmp_path):
    """No CPU fallback: without the CUDA library every entry point raises."""
    missing = str(tmp_path / "libmoe_layout.so")
    code = (
        "import sys\n"
        "from combine_moe_layout_05_gb300 import build, _binding\n"
        f"build.LIB_PATH = {missing!r}\n"
        "import combine_moe_layout_05_gb300 as moe\n"
        "for call in (lambda: moe.load(), lambda: moe.moe_layout_workspace_bytes(8, 2, 4)):\n"
        "    try:\n"
        "        call()\n"
        "    except RuntimeError as e:\n"
        "        assert 'missing' in str(e), e\n"
        "    else:\n"
        "        sys.exit('no error')\n"
    )
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr + r.stdout


def test_error_bits_agree_between_header_and_binding():
    import re
    text = open(os.path.join(ROOT, "include", "moe_layout.h")).read()
    bits = {m.group(1): int(m.group(2))
            for m in re.finditer(r"#define (MOE_DEV_ERR_\w+)\s+(\d+)u", text)}
    assert bits == {"MOE_DEV_ERR_EXPERT_RANGE": 1, "MOE_DEV_ERR_DUPLICATE": 2,
                    "MOE_DEV_ERR_REGION_OVERFLOW": 4, "MOE_DEV_ERR_TIMEOUT": 8}
    for name, v in bits.items():
        assert getattr(moe, name) == v, name
