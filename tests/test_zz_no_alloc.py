"""The no-allocation prefill entry point, gdn_chunk_fwd_staged_static.

It exists for callers that cannot allocate device memory (stream-capture or
host-callback code, allocators that own all device memory, hosts that hand
out only input and output buffers): it runs the staged prefill with its
scratch in one fixed array inside the library.  These tests call it through
the C ABI and check each result against the workspace-taking entry point
gdn_chunk_fwd_staged and against the fp64 oracle, within the tests' bf16
tolerance.  Consecutive calls use different problem sizes, so a call that
read what the previous one left in the shared array would be caught.  The
file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle

pytestmark = pytest.mark.gpu

TOL = 1e-2
GDN_ERR_SEQLENS, GDN_ERR_WORKSPACE = -4, -7


def _rel(x, ref):
    x = x.detach().double().cpu().numpy() if hasattr(x, "detach") else np.asarray(x, np.float64)
    ref = ref.detach().double().cpu().numpy() if hasattr(ref, "detach") else np.asarray(ref, np.float64)
    return float(np.max(np.abs(x - ref)) / max(float(np.max(np.abs(ref))), 1e-30))


def _entry(lib):
    f = lib.gdn_chunk_fwd_staged_static
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp]
    f.restype = ctypes.c_int
    return f


def _call_static(f, d, cu, n, T, H, D):
    """One call of the static entry; returns (o, h_T, device status)."""
    o = torch.full((T, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    hT = torch.full((n, H, D, D), float("nan"), device="cuda")
    st = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = f(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["log_alpha"].data_ptr(),
           d["beta"].data_ptr(), d["h0"].data_ptr(), cu.data_ptr(), n, T, H, D, D, 0, 1,
           o.data_ptr(), hT.data_ptr(), st.data_ptr(), stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    return o, hT, int(st.item())


def test_static_scratch_entry_matches_workspace_entry_and_oracle():
    import gated_deltanet_sequence_prefill_b300 as g
    f = _entry(g.lib)
    # a larger problem first, then a smaller one with other lengths, heads and values
    problems = [([900, 1, 513, 0, 330], 8, 21), ([300, 77, 0, 129], 4, 22)]
    for call, (lengths, H, seed) in enumerate(problems):
        D = 128
        inp = gi.gdn_inputs(lengths, H, D, D, "bf16", h0_std=0.01, seed=seed)
        d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
        T, n = sum(lengths), len(lengths)
        o, hT, status = _call_static(f, d, d["cu_seqlens"], n, T, H, D)
        assert status == 0, (call, status)
        o_ws, h_ws, ws = g.gdn_chunk_fwd_staged(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                                d["h0"], d["cu_seqlens"])
        assert g.workspace_status(ws) == 0
        assert _rel(o, o_ws) <= TOL and _rel(hT, h_ws) <= TOL, (call, _rel(o, o_ws), _rel(hT, h_ws))
        ro, rh = oracle.gdn(inp["q"], inp["k"], inp["v"], inp["log_alpha"], inp["beta"], inp["h0"],
                            inp["cu_seqlens"])
        assert _rel(o, ro) <= TOL and _rel(hT, rh) <= TOL, (call, _rel(o, ro), _rel(hT, rh))


def test_static_scratch_entry_reports_malformed_seqlens_then_recovers():
    import gated_deltanet_sequence_prefill_b300 as g
    f = _entry(g.lib)
    inp = gi.gdn_inputs([64, 64], 2, 128, 128, "bf16", h0_std=0.01, seed=23)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    bad = torch.tensor([0, 100, 64], dtype=torch.int32, device="cuda")  # decreasing
    _, _, status = _call_static(f, d, bad, 2, 128, 2, 128)
    assert status == GDN_ERR_SEQLENS
    o, hT, status = _call_static(f, d, d["cu_seqlens"], 2, 128, 2, 128)
    assert status == 0
    ro, rh = oracle.gdn(inp["q"], inp["k"], inp["v"], inp["log_alpha"], inp["beta"], inp["h0"],
                        inp["cu_seqlens"])
    assert _rel(o, ro) <= TOL and _rel(hT, rh) <= TOL


def test_static_scratch_entry_rejects_oversize_problems():
    import gated_deltanet_sequence_prefill_b300 as g
    f = _entry(g.lib)
    T, H, D = 131072, 32, 128
    assert g.staged_workspace_size(T, H, D, D, 1) > 64 << 20
    # rejected on the host before anything is read or launched
    rc = f(256, 256, 256, 256, 256, None, None, 1, T, H, D, D, 0, 1, 256, None, None, None)
    assert rc == GDN_ERR_WORKSPACE
