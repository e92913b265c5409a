"""Seeded synthetic inputs for GDN prefill, linear attention and decode.

This module holds input recipes only -- no arithmetic of the method -- and is
the one piece shared by the oracle-side tests and the CUDA-side callers.
All tensors are generated on the CPU with a seeded torch.Generator, so a
given (shape, seed) always yields the same values on any machine.

Recipe (distributions as stated for the workloads):
  q, k        ~ N(0,1) per element, L2-normalised per token in fp32 (x/||x||),
              then rounded once to the I/O dtype (bf16 round-to-nearest-even)
  v           ~ N(0,1), rounded once to the I/O dtype
  log_alpha   = -softplus(N(0,1)) * 0.1          (so alpha = exp(log_alpha) in (0,1))
  beta        = sigmoid(N(0,1))
  h0          ~ N(0, std=0.01) (fp32), or None
  linear attention: q, k = elu(N(0,1)) + 1 (feature map applied here, not in
              the kernel), v ~ N(0,1); no gates.
Gates are fp32 for prefill and bf16 for decode.
"""
import numpy as np
import torch
import torch.nn.functional as F

_DT = {"bf16": torch.bfloat16, "fp32": torch.float32}


def varlen_lengths(T, n_seqs, seed=0):
    """Split T tokens into n_seqs sequences: n_seqs-1 distinct cut points drawn
    uniformly from [1, T-1] with numpy's default_rng(seed), sorted."""
    if n_seqs == 1:
        return [T]
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, T), size=n_seqs - 1, replace=False))
    bounds = np.concatenate([[0], cuts, [T]])
    return [int(x) for x in np.diff(bounds)]


def cu_from_lengths(lengths):
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def _gen(seed):
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def _unit_rows(x):
    return x / x.norm(dim=-1, keepdim=True)


def gdn_inputs(lengths, H, dk, dv, dtype="bf16", h0_std=0.01, seed=0):
    """Packed varlen GDN prefill inputs (CPU tensors)."""
    g = _gen(seed)
    T = int(sum(lengths))
    dt = _DT[dtype]
    q = _unit_rows(torch.randn(T, H, dk, generator=g)).to(dt)
    k = _unit_rows(torch.randn(T, H, dk, generator=g)).to(dt)
    v = torch.randn(T, H, dv, generator=g).to(dt)
    log_alpha = (-F.softplus(torch.randn(T, H, generator=g)) * 0.1).float()
    beta = torch.sigmoid(torch.randn(T, H, generator=g)).float()
    h0 = None
    if h0_std:
        h0 = (torch.randn(len(lengths), H, dk, dv, generator=g) * h0_std).float()
    return dict(q=q, k=k, v=v, log_alpha=log_alpha, beta=beta, h0=h0,
                cu_seqlens=cu_from_lengths(lengths))


def linear_inputs(lengths, H, dk, dv, dtype="bf16", h0_std=0.0, seed=0):
    """Causal linear attention inputs with the elu+1 feature map applied."""
    g = _gen(seed)
    T = int(sum(lengths))
    dt = _DT[dtype]
    q = (F.elu(torch.randn(T, H, dk, generator=g)) + 1).to(dt)
    k = (F.elu(torch.randn(T, H, dk, generator=g)) + 1).to(dt)
    v = torch.randn(T, H, dv, generator=g).to(dt)
    h0 = None
    if h0_std:
        h0 = (torch.randn(len(lengths), H, dk, dv, generator=g) * h0_std).float()
    return dict(q=q, k=k, v=v, h0=h0, cu_seqlens=cu_from_lengths(lengths))


def decode_state(B, H, dk, dv, std=0.01, seed=0):
    """Initial fp32 decode state [B,H,dk,dv] (h = S^T)."""
    g = _gen(seed)
    return (torch.randn(B, H, dk, dv, generator=g) * std).float()


def decode_step_inputs(B, H, dk, dv, step, seed=0):
    """Inputs of one decode step (bf16 q,k,v,log_alpha,beta); each step has
    its own generator stream so any step can be regenerated alone."""
    g = _gen(1_000_003 * (int(seed) + 1) + int(step))
    q = _unit_rows(torch.randn(B, H, dk, generator=g)).to(torch.bfloat16)
    k = _unit_rows(torch.randn(B, H, dk, generator=g)).to(torch.bfloat16)
    v = torch.randn(B, H, dv, generator=g).to(torch.bfloat16)
    log_alpha = (-F.softplus(torch.randn(B, H, generator=g)) * 0.1).to(torch.bfloat16)
    beta = torch.sigmoid(torch.randn(B, H, generator=g)).to(torch.bfloat16)
    return dict(q=q, k=k, v=v, log_alpha=log_alpha, beta=beta)


# Workload shapes (sizes of the page-derived workloads)
WORKLOADS = {
    "gdn_fp32_small": dict(kind="gdn", lengths=[256], H=1, dk=64, dv=64, dtype="fp32", h0_std=0.0),
    "linear_b2_t4096": dict(kind="linear", lengths=[4096, 4096], H=8, dk=128, dv=128, dtype="bf16"),
    "gdn_t32k_h16": dict(kind="gdn", lengths=[32768], H=16, dk=128, dv=128, dtype="bf16", h0_std=0.01),
    "gdn_varlen_t128k_h32": dict(kind="gdn", lengths=varlen_lengths(131072, 4, 0), H=32, dk=128,
                                 dv=128, dtype="bf16", h0_std=0.01),
    "gdn_t128k_h32_single": dict(kind="gdn", lengths=[131072], H=32, dk=128, dv=128, dtype="bf16",
                                 h0_std=0.01),
    "decode_b128_h32": dict(kind="decode", B=128, H=32, dk=128, dv=128, steps=1024),
}
