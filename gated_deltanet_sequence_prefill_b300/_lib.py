"""ctypes binding of libgdn_b300.so: argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
checks tensor placement/dtype/contiguity, allocates outputs and workspaces
with PyTorch (the caller may pass its own), and forwards raw device pointers
and the current CUDA stream to the C entry points declared in include/gdn.h.
If the library is missing or older than its sources, importing this module
compiles it first (build.py, nvcc for sm_103a); if that fails, the import
raises: there is no fallback implementation.
"""
import ctypes
import os

import torch

from . import build as _build

LIB_PATH = _build.LIB

try:
    _build.build()
except Exception as e:  # no nvcc, or a compile error: no library, no package
    raise ImportError("libgdn_b300.so could not be built (%s): %s" % (LIB_PATH, e)) from e

lib = ctypes.CDLL(LIB_PATH)

_vp, _fp, _ip = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
_i, _i64, _sz = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t

GDN_BF16, GDN_FP32 = 0, 1
_PREFILL = [_vp, _vp, _vp, _fp, _fp, _fp, _ip, _i, _i64, _i, _i, _i, _i, _vp, _fp, _vp, _sz, _vp]
_SIZE = [_i64, _i, _i, _i, _i, _i]

lib.gdn_status_string.argtypes = [_i]
lib.gdn_status_string.restype = ctypes.c_char_p
lib.gdn_version.argtypes = []
lib.gdn_version.restype = ctypes.c_char_p
for _n in ("gdn_chunk_fwd_workspace_size", "linear_attn_fwd_workspace_size", "gdn_staged_workspace_size"):
    getattr(lib, _n).argtypes = _SIZE
    getattr(lib, _n).restype = _sz
lib.gdn_chunk_fwd.argtypes = _PREFILL
lib.gdn_chunk_fwd.restype = _i
lib.gdn_chunk_fwd_block_adjacent.argtypes = _PREFILL
lib.gdn_chunk_fwd_block_adjacent.restype = _i
lib.linear_attn_fwd.argtypes = [_vp, _vp, _vp, _fp, _ip, _i, _i64, _i, _i, _i, _i, _vp, _fp, _vp, _sz, _vp]
lib.linear_attn_fwd.restype = _i
lib.gdn_chunk_fwd_staged.argtypes = _PREFILL[:13] + [_i] + _PREFILL[13:]
lib.gdn_chunk_fwd_staged.restype = _i
lib.gdn_chunk_prepare.argtypes = [_vp, _vp, _fp, _fp, _ip, _i, _i64, _i, _i, _i, _i,
                                  _fp, _fp, _fp, _fp, _vp, _sz, _vp]
lib.gdn_chunk_prepare.restype = _i
lib.gdn_recurrent_step.argtypes = [_vp, _vp, _vp, _vp, _vp, _fp, _vp, _i, _i, _i, _i, _vp]
lib.gdn_recurrent_step.restype = _i
lib.gdn_workspace_status.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_int)]
lib.gdn_workspace_status.restype = _i
lib.gdn_workspace_timeout_site.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_int)]
lib.gdn_workspace_timeout_site.restype = _i
lib.linear_attn_variant_workspace_size.argtypes = [_i64, _i, _i, _i, _i, _i, _i, _i]
lib.linear_attn_variant_workspace_size.restype = _sz
lib.linear_attn_variant_fwd.argtypes = [_vp, _vp, _vp, _ip, _i, _i64, _i, _i, _i, _i, _i, _i, _vp, _fp,
                                        _fp, _vp, _sz, _vp]
lib.linear_attn_variant_fwd.restype = _i
lib.gdn_prefill_segments.argtypes = [_i64, _i, _i, _i, _i, _i, _i]
lib.gdn_prefill_segments.restype = _i
lib.gdn_set_wait_limit.argtypes = [_i]
lib.gdn_set_wait_limit.restype = _i

CHUNK = 64


class GdnError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (%d)" % (where, lib.gdn_status_string(status).decode(), status))


def _check(rc, where):
    if rc != 0:
        raise GdnError(rc, where)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(t, stream):
    if stream is not None:
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    return torch.cuda.current_stream(t.device).cuda_stream


def _io(t):
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_FP32
    raise TypeError("q/k/v must be bfloat16 or float32, got %s" % t.dtype)


def _need(t, name, dtype=None, ndim=None, device=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dims" % (name, ndim))
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))


def _prefill_shapes(q, k, v, cu_seqlens):
    T, H, dk = q.shape
    dv = v.shape[2]
    if k.shape != (T, H, dk) or v.shape[:2] != (T, H):
        raise ValueError("q/k/v shapes disagree")
    n_seqs = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    return T, H, dk, dv, n_seqs


def version():
    return lib.gdn_version().decode()


def status_string(s):
    return lib.gdn_status_string(int(s)).decode()


def chunk_fwd_workspace_size(T, H, dk, dv, n_seqs, dtype=torch.bfloat16, delta_rule=True):
    io = GDN_BF16 if dtype == torch.bfloat16 else GDN_FP32
    f = lib.gdn_chunk_fwd_workspace_size if delta_rule else lib.linear_attn_fwd_workspace_size
    return int(f(T, H, dk, dv, n_seqs, io))


def staged_workspace_size(T, H, dk, dv, n_seqs, dtype=torch.bfloat16):
    io = GDN_BF16 if dtype == torch.bfloat16 else GDN_FP32
    return int(lib.gdn_staged_workspace_size(T, H, dk, dv, n_seqs, io))


def _alloc_ws(nbytes, dev, workspace):
    if workspace is not None:
        return workspace
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=dev)


def _outputs(q, v, n_seqs, H, dk, dv, o, h_T, output_final_state):
    if o is None:
        o = torch.empty(q.shape[0], H, dv, dtype=q.dtype, device=q.device)
    if h_T is None and output_final_state:
        h_T = torch.empty(n_seqs, H, dk, dv, dtype=torch.float32, device=q.device)
    return o, h_T


def _check_inputs(q, k, v, log_alpha, beta, h0, cu_seqlens):
    _need(q, "q", ndim=3)
    dev = q.device
    _need(k, "k", q.dtype, 3, dev)
    _need(v, "v", q.dtype, 3, dev)
    _need(log_alpha, "log_alpha", torch.float32, 2, dev)
    _need(beta, "beta", torch.float32, 2, dev)
    _need(h0, "h0", torch.float32, 4, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1, dev)


def gdn_chunk_fwd(q, k, v, log_alpha, beta, h0=None, cu_seqlens=None, *, o=None, h_T=None,
                  workspace=None, output_final_state=True, stream=None, block_adjacent=False):
    """GDN prefill through the C ABI; returns (o, h_T, workspace).
    block_adjacent=True calls gdn_chunk_fwd_block_adjacent (the approximate
    block-adjacent intra-chunk solver) instead."""
    _check_inputs(q, k, v, log_alpha, beta, h0, cu_seqlens)
    T, H, dk, dv, n = _prefill_shapes(q, k, v, cu_seqlens)
    o, h_T = _outputs(q, v, n, H, dk, dv, o, h_T, output_final_state)
    ws = _alloc_ws(lib.gdn_chunk_fwd_workspace_size(T, H, dk, dv, n, _io(q)), q.device, workspace)
    f = lib.gdn_chunk_fwd_block_adjacent if block_adjacent else lib.gdn_chunk_fwd
    rc = f(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(h0), _ptr(cu_seqlens), n,
           T, H, dk, dv, _io(q), _ptr(o), _ptr(h_T), _ptr(ws), ws.numel(), _stream(q, stream))
    _check(rc, "gdn_chunk_fwd_block_adjacent" if block_adjacent else "gdn_chunk_fwd")
    return o, h_T, ws


def linear_attn_fwd(q, k, v, h0=None, cu_seqlens=None, *, o=None, h_T=None, workspace=None,
                    output_final_state=True, stream=None):
    """Causal linear attention through the C ABI; returns (o, h_T, workspace)."""
    _check_inputs(q, k, v, None, None, h0, cu_seqlens)
    T, H, dk, dv, n = _prefill_shapes(q, k, v, cu_seqlens)
    o, h_T = _outputs(q, v, n, H, dk, dv, o, h_T, output_final_state)
    ws = _alloc_ws(lib.linear_attn_fwd_workspace_size(T, H, dk, dv, n, _io(q)), q.device, workspace)
    rc = lib.linear_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(h0), _ptr(cu_seqlens), n, T, H, dk,
                             dv, _io(q), _ptr(o), _ptr(h_T), _ptr(ws), ws.numel(),
                             _stream(q, stream))
    _check(rc, "linear_attn_fwd")
    return o, h_T, ws


def gdn_chunk_fwd_staged(q, k, v, log_alpha=None, beta=None, h0=None, cu_seqlens=None, *,
                         delta_rule=True, o=None, h_T=None, workspace=None,
                         output_final_state=True, stream=None):
    """The three-kernel staged prefill; returns (o, h_T, workspace)."""
    _check_inputs(q, k, v, log_alpha, beta, h0, cu_seqlens)
    T, H, dk, dv, n = _prefill_shapes(q, k, v, cu_seqlens)
    o, h_T = _outputs(q, v, n, H, dk, dv, o, h_T, output_final_state)
    ws = _alloc_ws(lib.gdn_staged_workspace_size(T, H, dk, dv, n, _io(q)), q.device, workspace)
    rc = lib.gdn_chunk_fwd_staged(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                  _ptr(h0), _ptr(cu_seqlens), n, T, H, dk, dv, _io(q),
                                  int(bool(delta_rule)), _ptr(o), _ptr(h_T), _ptr(ws),
                                  ws.numel(), _stream(q, stream))
    _check(rc, "gdn_chunk_fwd_staged")
    return o, h_T, ws


def gdn_chunk_prepare(k, v, log_alpha, beta, cu_seqlens=None, n_chunks=None, *, workspace=None,
                      stream=None):
    """Intra-chunk stages only; returns (g, A, w, u, workspace), fp32.
    n_chunks (sum of ceil(L_s/64)) sizes A; by default its upper bound is used."""
    _check_inputs(k, k, v, log_alpha, beta, None, cu_seqlens)
    T, H, dk, dv, n = _prefill_shapes(k, k, v, cu_seqlens)
    if n_chunks is None:
        n_chunks = T // CHUNK + n
    dev = k.device
    g = torch.empty(T, H, dtype=torch.float32, device=dev)
    A = torch.zeros(max(n_chunks, 1), H, CHUNK, CHUNK, dtype=torch.float32, device=dev)
    w = torch.empty(T, H, dk, dtype=torch.float32, device=dev)
    u = torch.empty(T, H, dv, dtype=torch.float32, device=dev)
    ws = _alloc_ws(lib.gdn_staged_workspace_size(T, H, dk, dv, n, _io(k)), dev, workspace)
    rc = lib.gdn_chunk_prepare(_ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(cu_seqlens), n,
                               T, H, dk, dv, _io(k), _ptr(g), _ptr(A), _ptr(w), _ptr(u), _ptr(ws),
                               ws.numel(), _stream(k, stream))
    _check(rc, "gdn_chunk_prepare")
    return g, A[:n_chunks], w, u, ws


def gdn_recurrent_step(q, k, v, log_alpha, beta, state, *, o=None, stream=None):
    """One decode token, state [B,H,dk,dv] fp32 updated in place; returns o."""
    _need(q, "q", torch.bfloat16, 3)
    dev = q.device
    for name, t, nd in (("k", k, 3), ("v", v, 3), ("log_alpha", log_alpha, 2), ("beta", beta, 2)):
        _need(t, name, torch.bfloat16, nd, dev)
    _need(state, "state", torch.float32, 4, dev)
    B, H, dk = q.shape
    dv = v.shape[2]
    if o is None:
        o = torch.empty(B, H, dv, dtype=torch.bfloat16, device=dev)
    rc = lib.gdn_recurrent_step(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                _ptr(state), _ptr(o), B, H, dk, dv, _stream(q, stream))
    _check(rc, "gdn_recurrent_step")
    return o


def workspace_status(workspace, stream=None):
    """Synchronise the stream and read the workspace's device status word."""
    st = ctypes.c_int(0)
    _check(lib.gdn_workspace_status(_ptr(workspace), _stream(workspace, stream), ctypes.byref(st)),
           "gdn_workspace_status")
    return st.value


def workspace_timeout_site(workspace, stream=None):
    """Synchronise the stream and read which barrier the call's first timed-out
    wait gave up on (0: none)."""
    site = ctypes.c_int(0)
    _check(lib.gdn_workspace_timeout_site(_ptr(workspace), _stream(workspace, stream),
                                          ctypes.byref(site)), "gdn_workspace_timeout_site")
    return site.value


def set_wait_limit(polls):
    """Polls a bounded device wait makes before it reports GDN_ERR_TIMEOUT, for
    calls launched from now on (process-wide); negative restores the default.
    Returns the previous bound."""
    return int(lib.gdn_set_wait_limit(int(polls)))


def two_level_segments(T, H, n_seqs, dk=128, dv=128, dtype=torch.bfloat16, delta_rule=True):
    """Segments per sequence a prefill call of these sizes takes (1: one pass)."""
    io = GDN_BF16 if dtype == torch.bfloat16 else GDN_FP32
    return int(lib.gdn_prefill_segments(T, H, dk, dv, n_seqs, io, int(bool(delta_rule))))


def linear_attn_variant(q, k, v, cu_seqlens=None, *, causal=True, normalize=False, o=None,
                        output_kv=False, output_z=False, workspace=None, stream=None):
    """Linear attention, causal or bidirectional, optionally normalised, through
    the C ABI; returns (o, kv, z, workspace) with kv = K^T V [N,H,dk,dv] and
    z = summed keys [N,H,dk] (fp32, None unless asked for)."""
    _check_inputs(q, k, v, None, None, None, cu_seqlens)
    T, H, dk, dv, n = _prefill_shapes(q, k, v, cu_seqlens)
    o, _ = _outputs(q, v, n, H, dk, dv, o, None, False)
    kv = torch.empty(n, H, dk, dv, dtype=torch.float32, device=q.device) if output_kv else None
    z = torch.empty(n, H, dk, dtype=torch.float32, device=q.device) if output_z else None
    need = lib.linear_attn_variant_workspace_size(T, H, dk, dv, n, _io(q), int(bool(causal)),
                                                  int(bool(normalize)))
    ws = _alloc_ws(need, q.device, workspace)
    rc = lib.linear_attn_variant_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), n, T, H, dk, dv,
                                     _io(q), int(bool(causal)), int(bool(normalize)), _ptr(o),
                                     _ptr(kv), _ptr(z), _ptr(ws), ws.numel(), _stream(q, stream))
    _check(rc, "linear_attn_variant_fwd")
    return o, kv, z, ws
