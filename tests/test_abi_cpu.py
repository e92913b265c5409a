"""CPU-only checks of the C ABI: the library loads, exports every entry point
declared in include/gdn.h, and rejects bad arguments on the host before any
CUDA call (nothing here launches a kernel)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def g():
    # importing the package compiles the library first when it is missing or stale
    import gated_deltanet_sequence_prefill_b300 as pkg
    return pkg


def declared_functions():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"#define GDN_API.*", "", src)
    return sorted(set(re.findall(r"GDN_API\s+[\w\s\*]*?\b(\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("gdn_chunk_fwd", "linear_attn_fwd", "gdn_recurrent_step", "gdn_status_string",
              "gdn_chunk_fwd_workspace_size", "gdn_workspace_status"):
        assert n in names


def test_library_exports_every_declared_symbol(g):
    out = subprocess.run(["nm", "-D", "--defined-only", g.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(g.lib, n)


def test_status_strings_and_version(g):
    assert g.version().endswith("sm_103a")
    for code in range(0, -10, -1):
        assert g.status_string(code) != "unknown status"
    assert g.status_string(-42) == "unknown status"


def test_workspace_queries(g):
    # bf16 128x128 keeps intermediates on-chip only if the fused kernel is built;
    # the staged query must cover g, A, w, u in fp32
    T, H, N = 131072, 32, 4
    staged = g.staged_workspace_size(T, H, 128, 128, N)
    assert staged >= 4 * (T * H * (1 + 128 + 128) + (T // 64 + N) * H * 64 * 64)
    # the fused cluster kernel needs the plan plus 192 KB of global scratch per
    # (sequence, head): six 32 KB slots for the solve SM's per-chunk outputs
    fused = g.chunk_fwd_workspace_size(T, H, 128, 128, N)
    assert N * H * 192 * 1024 <= fused < N * H * 192 * 1024 + (1 << 20)
    assert fused < staged
    assert g.staged_workspace_size(T, H, 96, 128, N) == 0
    assert g.staged_workspace_size(-1, H, 128, 128, N) == 0


L = None


def _call_fwd(g, **kw):
    a = dict(q=256, k=256, v=256, la=256, b=256, h0=None, cu=256, n=2, T=128, H=2, dk=128,
             dv=128, io=0, o=256, hT=256, ws=256, wsb=1 << 40, st=None)
    a.update(kw)
    return g.lib.gdn_chunk_fwd(a["q"], a["k"], a["v"], a["la"], a["b"], a["h0"], a["cu"], a["n"],
                               a["T"], a["H"], a["dk"], a["dv"], a["io"], a["o"], a["hT"], a["ws"],
                               a["wsb"], a["st"])


def test_host_argument_checks(g):
    # every case returns before anything touches the (fake) device pointers
    assert _call_fwd(g, dk=96) == -6                 # UNSUPPORTED
    assert _call_fwd(g, dv=32) == -6
    assert _call_fwd(g, io=7) == -5                  # DTYPE
    assert _call_fwd(g, T=-1) == -3                  # SHAPE
    assert _call_fwd(g, H=0) == -3
    assert _call_fwd(g, cu=None, n=2) == -3          # NULL cu_seqlens needs n_seqs == 1
    assert _call_fwd(g, q=None) == -1                # NULL
    assert _call_fwd(g, la=None) == -1
    assert _call_fwd(g, ws=None) == -7               # WORKSPACE
    assert _call_fwd(g, wsb=16) == -7
    assert _call_fwd(g, q=256 + 8) == -2             # ALIGN (16 bytes)
    assert _call_fwd(g, ws=256 + 16) == -2           # workspace 256-byte alignment
    assert _call_fwd(g, la=256 + 2) == -2
    # decode
    f = g.lib.gdn_recurrent_step
    assert f(256, 256, 256, 256, 256, 256, 256, 4, 2, 100, 128, None) == -6
    assert f(256, 256, 256, 256, 256, 256, 256, -1, 2, 128, 128, None) == -3
    assert f(None, 256, 256, 256, 256, 256, 256, 4, 2, 128, 128, None) == -1
    assert f(256, 256, 256 + 4, 256, 256, 256, 256, 4, 2, 128, 128, None) == -2
    assert f(256, 256, 256, 256, 256, 256, 256, 0, 2, 128, 128, None) == 0  # empty batch


def test_binding_rejects_cpu_tensors(g):
    import torch
    q = torch.zeros(4, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        g.gdn_chunk_fwd(q, q, q, torch.zeros(4, 1), torch.zeros(4, 1))


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "gated_deltanet_sequence_prefill_b300")
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle)|liboracle|gdn_oracle", re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                assert not pat.search(open(os.path.join(dirpath, f)).read()), f


def test_wait_limit_setter(g):
    # the bound is host state only: set, read back through the next set, restore
    default = g.set_wait_limit(0)
    assert default == 1 << 22
    assert g.set_wait_limit(12345) == 0
    assert g.set_wait_limit(-1) == 12345
    assert g.set_wait_limit(-1) == default


def test_workspace_query_covers_the_two_level_scan(g, monkeypatch):
    # few long chains: the query includes the scan's runs and maps
    T, H, N = 131072, 4, 1
    monkeypatch.setenv("GDN_TWO_LEVEL", "0")
    plain = g.chunk_fwd_workspace_size(T, H, 128, 128, N)
    monkeypatch.delenv("GDN_TWO_LEVEL")
    scan = g.chunk_fwd_workspace_size(T, H, 128, 128, N)
    assert plain < N * H * 192 * 1024 + (1 << 20)
    # G segments per sequence: cluster scratch plus M, B and h_start (64 KB each) per segment and head
    G = min(16, 37 // (N * H) + 1)
    assert scan >= N * G * H * (192 + 3 * 64) * 1024
    monkeypatch.setenv("GDN_TWO_LEVEL", "5")
    assert g.chunk_fwd_workspace_size(T, H, 128, 128, N) >= N * 5 * H * (192 + 3 * 64) * 1024
    # many chains: no scan
    monkeypatch.delenv("GDN_TWO_LEVEL")
    assert g.chunk_fwd_workspace_size(T, 32, 128, 128, 4) < 4 * 32 * 192 * 1024 + (1 << 20)
