"""fp64 CPU oracle for the gated delta rule (GDN) and causal linear attention.

TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import this package; the CUDA path neither
imports it nor shares any code with it.

What it computes (the readings are listed with the C source, gdn_oracle.c):
  gdn(...)        token-by-token gated delta rule
                  S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,  o_t = S_t q_t
  linear(...)     plain causal linear attention S_t = S_{t-1} + v_t k_t^T
                  ("Как ускорить LLM на длинном контексте", section "Linear attention")
  decode_step(.)  one token of the gated delta rule applied to a given state
  chunked(...)    the chunk-wise evaluation (intra-chunk delta-system solve,
                  sequential pass over chunks, outputs from chunk-start states:
                  SparseGDN article, "Чем дорог префилл в Gated Delta Networks…")
  linear_variant(...)  linear attention with the causal mask optional and the
                  normaliser optional: o_t = sum_s w_ts v_s with w_ts = q_t . k_s
                  over s <= t (causal) or all s of the sequence (bidirectional),
                  divided by sum_s w_ts when normalised (datadaily.news
                  "За пределами self-attention", section "Линейное внимание…",
                  the normalised listing; ai-vestnik.ru item on linear attention:
                  the bidirectional mode and the causal restriction).
  linear_quadratic(...)  the quadratic masked form (Q K^T ⊙ M) V + Q h0 of
                  causal linear attention (datadaily.news "За пределами
                  self-attention", section "Линейное внимание…": the two
                  evaluation orders of (φ(Q)φ(K)^T)V), M lower-triangular with
                  the diagonal included.

Arrays are token-major: q,k [T,H,dk], v [T,H,dv], log_alpha/beta [T,H],
h0/hT [N,H,dk,dv] with h = S^T.  Inputs may be numpy arrays or CPU torch
tensors of any float dtype; they are upcast to float64 exactly.
"""
import contextlib
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def _load(path):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int64)
    lib.oracle_recurrent.argtypes = [dp, dp, dp, dp, dp, dp, ip, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     dp, dp, ctypes.c_int]
    lib.oracle_recurrent.restype = ctypes.c_int
    lib.oracle_chunked.argtypes = [dp, dp, dp, dp, dp, dp, ip, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int]
    lib.oracle_chunked.restype = ctypes.c_int
    lib.oracle_chunked_band.argtypes = [dp, dp, dp, dp, dp, dp, ip, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, dp, dp, dp, dp, dp, dp, dp,
                                        ctypes.c_int]
    lib.oracle_chunked_band.restype = ctypes.c_int
    lib.oracle_num_chunks.argtypes = [ip, ctypes.c_int, ctypes.c_int]
    lib.oracle_num_chunks.restype = ctypes.c_int64
    lib.oracle_num_threads.argtypes = [ctypes.c_int]
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def _lib():
    global _LIB
    if _LIB is None:
        _LIB = _load(_build.build())
    return _LIB


@contextlib.contextmanager
def using_library(path):
    """Run the oracle from another build of its source while the context is
    open (the pins' planted-mistake tests load a deliberately broken copy)."""
    global _LIB
    saved = _LIB
    _LIB = _load(path)
    try:
        yield
    finally:
        _LIB = saved


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a, typ=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(typ))


def _cu(cu_seqlens, T):
    if cu_seqlens is None:
        return np.array([0, T], dtype=np.int64)
    if hasattr(cu_seqlens, "detach"):
        cu_seqlens = cu_seqlens.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))


def _check(rc):
    if rc != 0:
        raise ValueError("oracle error %d" % rc)


def num_threads(n=0):
    return _lib().oracle_num_threads(n)


def recurrent(q, k, v, log_alpha=None, beta=None, h0=None, cu_seqlens=None,
              delta_rule=True, threads=0):
    """Token-by-token recurrence; returns (o [T,H,dv], hT [N,H,dk,dv]) in float64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    la, b, h0 = _f64(log_alpha), _f64(beta), _f64(h0)
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = _cu(cu_seqlens, T)
    N = len(cu) - 1
    if cu[-1] != T:
        raise ValueError("cu_seqlens[-1] != T")
    o = np.zeros((T, H, dv))
    hT = np.zeros((N, H, dk, dv))
    rc = _lib().oracle_recurrent(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b), _ptr(h0),
                                 _ptr(cu, ctypes.c_int64), N, H, dk, dv, int(bool(delta_rule)),
                                 _ptr(o), _ptr(hT), int(threads))
    _check(rc)
    return o, hT


def gdn(q, k, v, log_alpha, beta, h0=None, cu_seqlens=None, threads=0):
    """Gated delta rule prefill, token by token (the definition)."""
    return recurrent(q, k, v, log_alpha, beta, h0, cu_seqlens, True, threads)


def linear(q, k, v, h0=None, cu_seqlens=None, threads=0):
    """Plain causal linear attention S_t = S_{t-1} + v_t k_t^T, o_t = S_t q_t."""
    return recurrent(q, k, v, None, None, h0, cu_seqlens, False, threads)


def decode_step(q, k, v, log_alpha, beta, state, threads=0):
    """One gated-delta-rule token per (sequence, head): q,k [B,H,dk], v [B,H,dv],
    log_alpha/beta [B,H], state [B,H,dk,dv] (h = S^T).  Returns (o, new_state)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B = q.shape[0]
    cu = np.arange(B + 1, dtype=np.int64)
    return recurrent(q, k, v, log_alpha, beta, state, cu, True, threads)


def num_chunks(cu_seqlens, chunk):
    cu = _cu(cu_seqlens, None)
    return int(_lib().oracle_num_chunks(_ptr(cu, ctypes.c_int64), len(cu) - 1, chunk))


def chunked(q, k, v, log_alpha=None, beta=None, h0=None, cu_seqlens=None, chunk=64,
            delta_rule=True, intermediates=False, threads=0, band=0):
    """Chunk-wise evaluation.  Returns (o, hT) or, with intermediates=True,
    (o, hT, dict(A, Tm, w, u, g)) where A/Tm are [n_chunks, H, C, C].
    band > 0: the block-adjacent solver (Tm kept on the diagonal blocks of
    `band` tokens and the blocks right below them; SparseGDN article,
    "Двухуровневая разреженность SparseGDN…")."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    la, b, h0 = _f64(log_alpha), _f64(beta), _f64(h0)
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = _cu(cu_seqlens, T)
    N = len(cu) - 1
    if cu[-1] != T:
        raise ValueError("cu_seqlens[-1] != T")
    o = np.zeros((T, H, dv))
    hT = np.zeros((N, H, dk, dv))
    inter = None
    A = Tm = w = u = g = None
    if intermediates:
        nch = num_chunks(cu, chunk)
        A = np.zeros((nch, H, chunk, chunk))
        Tm = np.zeros((nch, H, chunk, chunk))
        w = np.zeros((T, H, dk))
        u = np.zeros((T, H, dv))
        g = np.zeros((T, H))
        inter = dict(A=A, Tm=Tm, w=w, u=u, g=g)
    if band:
        rc = _lib().oracle_chunked_band(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b), _ptr(h0),
                                        _ptr(cu, ctypes.c_int64), N, H, dk, dv, int(chunk),
                                        int(bool(delta_rule)), int(band), _ptr(o), _ptr(hT),
                                        _ptr(A), _ptr(Tm), _ptr(w), _ptr(u), _ptr(g), int(threads))
    else:
        rc = _lib().oracle_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b), _ptr(h0),
                                   _ptr(cu, ctypes.c_int64), N, H, dk, dv, int(chunk),
                                   int(bool(delta_rule)), _ptr(o), _ptr(hT), _ptr(A), _ptr(Tm),
                                   _ptr(w), _ptr(u), _ptr(g), int(threads))
    _check(rc)
    if intermediates:
        return o, hT, inter
    return o, hT


def linear_quadratic(q, k, v, h0=None, cu_seqlens=None):
    """Quadratic masked form of causal linear attention, per sequence and head:
    O = (Q K^T ⊙ M) V + Q h0, M[i][j] = 1 for j <= i.  Also returns
    hT = h0 + K^T V.  (Q h0 = (S0 q_t)^T per row, with h0 = S0^T.)"""
    q, k, v, h0 = _f64(q), _f64(k), _f64(v), _f64(h0)
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = _cu(cu_seqlens, T)
    N = len(cu) - 1
    o = np.zeros((T, H, dv))
    hT = np.zeros((N, H, dk, dv))
    for s in range(N):
        a, e = int(cu[s]), int(cu[s + 1])
        for h in range(H):
            Q, K, V = q[a:e, h], k[a:e, h], v[a:e, h]
            M = np.tril(np.ones((e - a, e - a)))
            out = (Q @ K.T * M) @ V
            st = K.T @ V
            if h0 is not None:
                out = out + Q @ h0[s, h]
                st = st + h0[s, h]
            o[a:e, h] = out
            hT[s, h] = st
    return o, hT


def linear_variant(q, k, v, cu_seqlens=None, causal=True, normalize=False):
    """Linear attention in its quadratic form, per sequence and head, fp64:
        W = Q K^T, masked to s <= t when causal (diagonal included);
        o = W V, divided row by row by W 1 when normalised.
    Also returns, per sequence and head, kv = K^T V (dk x dv, the summed
    state) and z = K^T 1 (the summed keys).  The feature map (elu + 1 on the
    page) is applied by the caller to q and k beforehand; no epsilon is added
    to the normaliser (the page adds none)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = _cu(cu_seqlens, T)
    N = len(cu) - 1
    o = np.zeros((T, H, dv))
    kv = np.zeros((N, H, dk, dv))
    z = np.zeros((N, H, dk))
    for s in range(N):
        a, e = int(cu[s]), int(cu[s + 1])
        for h in range(H):
            Q, K, V = q[a:e, h], k[a:e, h], v[a:e, h]
            W = Q @ K.T
            if causal:
                W = W * np.tril(np.ones((e - a, e - a)))
            out = W @ V
            if normalize:
                out = out / W.sum(axis=1, keepdims=True)
            o[a:e, h] = out
            kv[s, h] = K.T @ V
            z[s, h] = K.sum(axis=0)
    return o, kv, z


def linear_sums(k, v, cu_seqlens=None):
    """Per sequence and head, kv = K^T V and z = K^T 1 (fp64): the aggregates
    the bidirectional form reassociates through (same page and listing as
    linear_variant), without the T x T weights, for long inputs."""
    k, v = _f64(k), _f64(v)
    T, H, dk = k.shape
    dv = v.shape[2]
    cu = _cu(cu_seqlens, T)
    N = len(cu) - 1
    kv = np.zeros((N, H, dk, dv))
    z = np.zeros((N, H, dk))
    for s in range(N):
        a, e = int(cu[s]), int(cu[s + 1])
        for h in range(H):
            kv[s, h] = k[a:e, h].T @ v[a:e, h]
            z[s, h] = k[a:e, h].sum(axis=0)
    return kv, z
