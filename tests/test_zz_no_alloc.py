"""The no-allocation prefill entry point, gdn_chunk_fwd_staged_static.

It exists for callers that cannot allocate device memory (stream-capture or
host-callback code, allocators that own all device memory, hosts that hand
out only input and output buffers): it runs the staged prefill with its
scratch in one fixed array inside the library.  This test calls it through
the C ABI twice in a row and checks each result against the workspace-taking
entry point gdn_chunk_fwd_staged, within the tests' bf16 tolerance.  The file
name sorts last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import pytest
import torch

import gdn_inputs as gi

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _rel(x, ref):
    x, ref = x.double(), ref.double()
    return float((x - ref).abs().max() / ref.abs().max().clamp_min(1e-30))


def _entry(lib):
    f = lib.gdn_chunk_fwd_staged_static
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp]
    f.restype = ctypes.c_int
    return f


def test_static_scratch_entry_matches_workspace_entry():
    import gated_deltanet_sequence_prefill_b300 as g
    f = _entry(g.lib)
    lengths = [300, 77, 0, 129]
    H, D = 4, 128
    inp = {k: (v.cuda() if v is not None else None)
           for k, v in gi.gdn_inputs(lengths, H, D, D, "bf16", h0_std=0.01, seed=21).items()}
    T, n = sum(lengths), len(lengths)
    o_ref, h_ref, ws = g.gdn_chunk_fwd_staged(inp["q"], inp["k"], inp["v"], inp["log_alpha"],
                                              inp["beta"], inp["h0"], inp["cu_seqlens"])
    assert g.workspace_status(ws) == 0
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        o = torch.full((T, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        hT = torch.full((n, H, D, D), float("nan"), device="cuda")
        st = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
        rc = f(inp["q"].data_ptr(), inp["k"].data_ptr(), inp["v"].data_ptr(),
               inp["log_alpha"].data_ptr(), inp["beta"].data_ptr(), inp["h0"].data_ptr(),
               inp["cu_seqlens"].data_ptr(), n, T, H, D, D, 0, 1, o.data_ptr(), hT.data_ptr(),
               st.data_ptr(), stream)
        assert rc == 0, g.status_string(rc)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, call
        assert _rel(o, o_ref) <= TOL, (call, _rel(o, o_ref))
        assert _rel(hT, h_ref) <= TOL, (call, _rel(hT, h_ref))


def test_static_scratch_entry_rejects_oversize_problems():
    import gated_deltanet_sequence_prefill_b300 as g
    f = _entry(g.lib)
    T, H, D = 131072, 32, 128
    assert g.staged_workspace_size(T, H, D, D, 1) > 64 << 20
    # rejected on the host before anything is read or launched (GDN_ERR_WORKSPACE)
    rc = f(256, 256, 256, 256, 256, None, None, 1, T, H, D, D, 0, 1, 256, None, None, None)
    assert rc == -7
