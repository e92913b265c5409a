"""GPU parity: the CUDA path (called through the C ABI) against the fp64
oracle on the same seeded inputs.

Tolerance (stated for this method): max|x - x_ref| / max|x_ref| over the
whole compared tensor, <= 1e-2 for bf16 I/O with fp32 accumulation and
<= 1e-4 for fp32 I/O, applied separately to o and to the final state h_T.
"""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "fp32": 1e-4}


@pytest.fixture(scope="module")
def g():
    import gated_deltanet_sequence_prefill_b300 as pkg
    assert torch.cuda.is_available()
    return pkg


def rel(x, ref):
    if hasattr(x, "detach"):
        x = x.detach().double().cpu().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(x - ref)) / max(float(np.max(np.abs(ref))), 1e-30))


def dev(inp):
    return {k: (v.cuda() if v is not None else None) for k, v in inp.items()}


def run_gdn(g, inp, staged=False, **kw):
    d = dev(inp)
    f = g.gdn_chunk_fwd_staged if staged else g.gdn_chunk_fwd
    o, hT, ws = f(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["h0"], d["cu_seqlens"], **kw)
    st = g.workspace_status(ws)
    assert st == 0, g.status_string(st)
    return o, hT


def ref_gdn(inp, chains=None):
    """Oracle on all chains, or on the (seq, head) pairs in `chains`."""
    if chains is None:
        return oracle.gdn(inp["q"], inp["k"], inp["v"], inp["log_alpha"], inp["beta"],
                          inp["h0"], inp["cu_seqlens"])
    cu = inp["cu_seqlens"].tolist()
    out = {}
    for s, h in chains:
        a, e = cu[s], cu[s + 1]
        h0 = None if inp["h0"] is None else inp["h0"][s:s + 1, h:h + 1]
        o, hT = oracle.gdn(inp["q"][a:e, h:h + 1], inp["k"][a:e, h:h + 1], inp["v"][a:e, h:h + 1],
                           inp["log_alpha"][a:e, h:h + 1], inp["beta"][a:e, h:h + 1], h0)
        out[(s, h)] = (o[:, 0], hT[0, 0])
    return out


def ref_heads(inp, chains):
    """Oracle on the sampled (seq, head) chains, one call per sequence so that
    its threads run the sampled heads of that sequence in parallel."""
    cu = inp["cu_seqlens"].tolist()
    out = {}
    for s in sorted({c[0] for c in chains}):
        hs = [h for (s2, h) in chains if s2 == s]
        a, e = cu[s], cu[s + 1]
        h0 = None if inp["h0"] is None else inp["h0"][s:s + 1, hs]
        o, hT = oracle.gdn(inp["q"][a:e, hs], inp["k"][a:e, hs], inp["v"][a:e, hs],
                           inp["log_alpha"][a:e, hs], inp["beta"][a:e, hs], h0)
        for i, h in enumerate(hs):
            out[(s, h)] = (o[:, i], hT[0, i])
    return out


def check_chains(inp, o, hT, chains, tol):
    ref = ref_heads(inp, chains)
    cu = inp["cu_seqlens"].tolist()
    o_got = np.concatenate([o[cu[s]:cu[s + 1], h].double().cpu().numpy() for s, h in chains])
    o_ref = np.concatenate([ref[c][0] for c in chains])
    h_got = np.stack([hT[s, h].double().cpu().numpy() for s, h in chains])
    h_ref = np.stack([ref[c][1] for c in chains])
    assert rel(o_got, o_ref) <= tol, rel(o_got, o_ref)
    assert rel(h_got, h_ref) <= tol, rel(h_got, h_ref)


# ------------------------------------------------------------------ small / ragged

def test_gdn_fp32_t256_d64(g):
    """GDN, one sequence of 256 tokens, one head, dk = dv = 64, fp32 I/O."""
    inp = gi.gdn_inputs([256], 1, 64, 64, "fp32", h0_std=0.0, seed=0)
    o, hT = run_gdn(g, inp)
    ro, rh = ref_gdn(inp)
    assert rel(o, ro) <= TOL["fp32"] and rel(hT, rh) <= TOL["fp32"], (rel(o, ro), rel(hT, rh))


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("staged", [False, True])
def test_gdn_ragged_varlen(g, dk, dv, dtype, staged):
    lengths = [1, 70, 0, 129, 64, 200, 63]
    inp = gi.gdn_inputs(lengths, 3, dk, dv, dtype, h0_std=0.01, seed=1)
    o, hT = run_gdn(g, inp, staged=staged)
    ro, rh = ref_gdn(inp)
    assert rel(o, ro) <= TOL[dtype], rel(o, ro)
    assert rel(hT, rh) <= TOL[dtype], rel(hT, rh)


# (GDN_PREFILL_PAIR, GDN_PREFILL_FRONTS): the cluster kernel with one or two
# solve CTAs per cluster, and the single-SM kernel
KERNELS = [pytest.param(("1", "1"), id="pair_1solve"), pytest.param(("1", "2"), id="pair_2solve"),
           pytest.param(("0", None), id="single_sm")]


def use_kernel(monkeypatch, kernel):
    monkeypatch.setenv("GDN_LINEAR_PATH", "cluster")  # linear attention through the fused kernels too
    monkeypatch.setenv("GDN_PREFILL_PAIR", kernel[0])
    if kernel[1] is None:
        monkeypatch.delenv("GDN_PREFILL_FRONTS", raising=False)
    else:
        monkeypatch.setenv("GDN_PREFILL_FRONTS", kernel[1])


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("scale", [6.0, 40.0])
def test_gdn_strong_gates(g, monkeypatch, kernel, scale):
    """Strongly negative log-decays: a chunk's decay range (about 30 at scale
    6, about 200 at scale 40) straddles or passes the limit of the factored
    form, so both decay paths of each fused kernel run."""
    use_kernel(monkeypatch, kernel)
    inp = gi.gdn_inputs([700, 333, 129], 4, 128, 128, "bf16", h0_std=0.5, seed=5)
    inp["log_alpha"] = inp["log_alpha"] * scale
    o, hT = run_gdn(g, inp)
    ro, rh = ref_gdn(inp)
    assert rel(o, ro) <= TOL["bf16"], rel(o, ro)
    assert rel(hT, rh) <= TOL["bf16"], rel(hT, rh)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("lengths,h0_std", [([1, 70, 0, 129, 64, 200, 63], 0.01), ([700, 333], 0.5)])
def test_fused_kernels(g, monkeypatch, kernel, lengths, h0_std):
    """Each fused kernel, forced through the environment, against the oracle
    on ragged packed sequences (the automatic choice picks the cluster kernel
    for these few units)."""
    use_kernel(monkeypatch, kernel)
    inp = gi.gdn_inputs(lengths, 4, 128, 128, "bf16", h0_std=h0_std, seed=3)
    o, hT = run_gdn(g, inp)
    ro, rh = ref_gdn(inp)
    assert rel(o, ro) <= TOL["bf16"], rel(o, ro)
    assert rel(hT, rh) <= TOL["bf16"], rel(hT, rh)


@pytest.mark.parametrize("seed", [1, 2])
def test_gdn_seeds(g, seed):
    inp = gi.gdn_inputs([300, 777], 4, 128, 128, "bf16", h0_std=0.01, seed=seed)
    o, hT = run_gdn(g, inp)
    ro, rh = ref_gdn(inp)
    assert rel(o, ro) <= TOL["bf16"] and rel(hT, rh) <= TOL["bf16"]


def test_prepare_intermediates_match_oracle(g):
    """Stages 1-2 alone: chunk gate sums g, A, and the WY pair w, u."""
    lengths = [70, 129, 5]
    inp = gi.gdn_inputs(lengths, 2, 64, 128, "fp32", h0_std=0.0, seed=3)
    d = dev(inp)
    n_chunks = oracle.num_chunks(inp["cu_seqlens"], 64)
    gg, A, w, u, ws = g.gdn_chunk_prepare(d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"],
                                          n_chunks=n_chunks)
    assert g.workspace_status(ws) == 0
    _, _, it = oracle.chunked(inp["q"], inp["k"], inp["v"], inp["log_alpha"], inp["beta"], None,
                              inp["cu_seqlens"], chunk=64, intermediates=True)
    assert rel(gg, it["g"]) <= 1e-5
    assert rel(A, it["A"]) <= 1e-4
    assert rel(w, it["w"]) <= 1e-4
    assert rel(u, it["u"]) <= 1e-4


# ------------------------------------------------------------------ workload sizes

def test_linear_b2_t4096_h8(g):
    """Plain causal linear attention, 2 x 4096 tokens, H = 8, d = 128, bf16;
    against the token recurrence and the quadratic masked form."""
    inp = gi.linear_inputs([4096, 4096], 8, 128, 128, "bf16", seed=0)
    d = dev(inp)
    o, hT, ws = g.linear_attn_fwd(d["q"], d["k"], d["v"], None, d["cu_seqlens"])
    assert g.workspace_status(ws) == 0
    ro, rh = oracle.linear(inp["q"], inp["k"], inp["v"], None, inp["cu_seqlens"])
    qo, qh = oracle.linear_quadratic(inp["q"], inp["k"], inp["v"], None, inp["cu_seqlens"])
    assert rel(ro, qo) < 1e-10
    assert rel(o, ro) <= TOL["bf16"] and rel(hT, rh) <= TOL["bf16"]
    assert rel(o, qo) <= TOL["bf16"] and rel(hT, qh) <= TOL["bf16"]


@pytest.mark.parametrize("kernel", KERNELS)
def test_linear_ragged_with_h0(g, monkeypatch, kernel):
    """Ragged linear attention with an initial state through each fused kernel
    (the gate-free instantiation: T is the identity, P^ is the causal q k^T)."""
    use_kernel(monkeypatch, kernel)
    inp = gi.linear_inputs([1, 100, 0, 257], 4, 128, 128, "bf16", h0_std=0.5, seed=4)
    d = dev(inp)
    o, hT, ws = g.linear_attn_fwd(d["q"], d["k"], d["v"], d["h0"], d["cu_seqlens"])
    assert g.workspace_status(ws) == 0
    ro, rh = oracle.linear(inp["q"], inp["k"], inp["v"], inp["h0"], inp["cu_seqlens"])
    assert rel(o, ro) <= TOL["bf16"] and rel(hT, rh) <= TOL["bf16"]


def test_gdn_t32768_h16(g):
    """GDN prefill, one 32768-token sequence, H = 16, d = 128, bf16 I/O;
    oracle on a sample of heads (every token of each)."""
    inp = gi.gdn_inputs([32768], 16, 128, 128, "bf16", h0_std=0.01, seed=0)
    o, hT = run_gdn(g, inp)
    check_chains(inp, o, hT, [(0, 0), (0, 5), (0, 11), (0, 15)], TOL["bf16"])


@pytest.mark.parametrize("fronts", ["1", "2"])
def test_pair_kernel_varlen_t131072_h32(g, monkeypatch, fronts):
    """The cluster kernel with one or two solve CTAs, forced, on the
    benchmarked packed call (128 clusters, more than fit at once): 8 sampled
    chains against the oracle."""
    monkeypatch.setenv("GDN_PREFILL_PAIR", "1")
    monkeypatch.setenv("GDN_PREFILL_FRONTS", fronts)
    lengths = gi.varlen_lengths(131072, 4, 0)
    inp = gi.gdn_inputs(lengths, 32, 128, 128, "bf16", h0_std=0.01, seed=0)
    o, hT = run_gdn(g, inp)
    chains = [(0, 0), (0, 31), (1, 5), (2, 17), (3, 9), (3, 30), (1, 22), (2, 2)]
    check_chains(inp, o, hT, chains, TOL["bf16"])


def test_gdn_varlen_t131072_h32(g):
    """GDN long prefill, 4 packed sequences (seeded lengths) summing to 131072
    tokens, H = 32, d = 128, bf16: the benchmarked call.  Oracle on 8 sampled
    (sequence, head) chains, every token of each, and their final states."""
    lengths = gi.varlen_lengths(131072, 4, 0)
    inp = gi.gdn_inputs(lengths, 32, 128, 128, "bf16", h0_std=0.01, seed=0)
    o, hT = run_gdn(g, inp)
    assert torch.isfinite(o.float()).all() and torch.isfinite(hT).all()
    check_chains(inp, o, hT, [(0, 0), (0, 31), (1, 7), (1, 20), (2, 3), (2, 16), (3, 9), (3, 30)],
                 TOL["bf16"])


@pytest.mark.parametrize("staged", [False, True])
def test_fused_and_staged_t32768_against_oracle(g, staged):
    """gdn_chunk_fwd and the staged three-kernel path, each against the oracle
    on a full-size two-sequence input (sampled chains, every token of each)."""
    inp = gi.gdn_inputs([20000, 12768], 16, 128, 128, "bf16", h0_std=0.01, seed=5)
    o, hT = run_gdn(g, inp, staged=staged)
    check_chains(inp, o, hT, [(0, 0), (0, 9), (0, 15), (1, 3), (1, 12)], TOL["bf16"])


def test_gdn_single_sequence_t131072_h32(g):
    """The hardest chain: one 131072-token sequence, H = 32 (the automatic
    choice runs the cluster kernel with two solve CTAs per cluster at full
    length).  Oracle on sampled heads, every token of each, and h_T."""
    inp = gi.gdn_inputs([131072], 32, 128, 128, "bf16", h0_std=0.01, seed=0)
    o, hT = run_gdn(g, inp)
    assert torch.isfinite(o.float()).all() and torch.isfinite(hT).all()
    check_chains(inp, o, hT, [(0, 0), (0, 13), (0, 22), (0, 31)], TOL["bf16"])


# ------------------------------------------------------------------ block-adjacent solver

def ref_band(inp, **kw):
    return oracle.chunked(inp["q"], inp["k"], inp["v"], inp["log_alpha"], inp["beta"], inp["h0"],
                          inp["cu_seqlens"], band=16, **kw)


@pytest.mark.parametrize("dk,dv,dtype", [(64, 64, "fp32"), (128, 128, "fp32"), (64, 128, "fp32"),
                                         (128, 64, "bf16"), (128, 128, "bf16")])
def test_block_adjacent_against_oracle(g, dk, dv, dtype):
    """gdn_chunk_fwd_block_adjacent against the oracle's block-adjacent solve
    (16-token blocks), at the dtype's tolerance; the approximation itself is
    far outside that tolerance from the exact solve on these inputs, so the
    comparison tells the two apart."""
    inp = gi.gdn_inputs([300, 77, 0, 129, 1], 4, dk, dv, dtype, h0_std=0.01, seed=31)
    o, hT = run_gdn(g, inp, block_adjacent=True)
    ob, hb = ref_band(inp)
    assert rel(o, ob) <= TOL[dtype], rel(o, ob)
    assert rel(hT, hb) <= TOL[dtype], rel(hT, hb)
    oe, _ = ref_gdn(inp)
    assert rel(ob, oe) > 2 * TOL[dtype]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("scale", [1.0, 40.0])
def test_block_adjacent_fused_kernels(g, monkeypatch, kernel, scale):
    """The block-adjacent solve in each fused kernel (ordinary gates, and
    strong ones that take the kernels' large-decay path)."""
    use_kernel(monkeypatch, kernel)
    inp = gi.gdn_inputs([700, 63, 200], 4, 128, 128, "bf16", h0_std=0.01, seed=32)
    inp["log_alpha"] = inp["log_alpha"] * scale
    o, hT = run_gdn(g, inp, block_adjacent=True)
    ob, hb = ref_band(inp)
    assert rel(o, ob) <= TOL["bf16"] and rel(hT, hb) <= TOL["bf16"], (rel(o, ob), rel(hT, hb))


def test_block_adjacent_varlen_t131072_h32(g):
    """The benchmarked packed call (4 sequences, 131072 tokens, H = 32) with
    the block-adjacent solve; every token of sampled heads of the shortest
    sequence against the oracle's banded solve, and their final states."""
    lengths = gi.varlen_lengths(131072, 4, 0)
    inp = gi.gdn_inputs(lengths, 32, 128, 128, "bf16", h0_std=0.01, seed=0)
    o, hT = run_gdn(g, inp, block_adjacent=True)
    s = int(np.argmin(lengths))
    cu = inp["cu_seqlens"].tolist()
    a, e = cu[s], cu[s + 1]
    hs = [0, 11, 31]
    sub = {k: inp[k][a:e, hs] for k in ("q", "k", "v", "log_alpha", "beta")}
    sub["h0"] = inp["h0"][s:s + 1, hs]
    sub["cu_seqlens"] = None
    ob, hb = ref_band(sub)
    assert rel(o[a:e, hs], ob) <= TOL["bf16"] and rel(hT[s, hs], hb[0]) <= TOL["bf16"]


# ------------------------------------------------------------------ two-level state scan

@pytest.mark.parametrize("G", ["2", "5"])
@pytest.mark.parametrize("delta", [True, False])
def test_two_level_scan_against_oracle(g, monkeypatch, G, delta):
    """The two-level state scan forced to G segments per sequence (transition
    maps and offsets of all segments side by side, a scan of the maps, then
    the outputs from the segment starts) on ragged packed sequences: every
    token and every final state against the oracle."""
    monkeypatch.setenv("GDN_TWO_LEVEL", G)
    lengths = [700, 1, 0, 333, 2000]
    if delta:
        inp = gi.gdn_inputs(lengths, 4, 128, 128, "bf16", h0_std=0.01, seed=41)
        o, hT = run_gdn(g, inp)
        ro, rh = ref_gdn(inp)
    else:
        inp = gi.linear_inputs(lengths, 4, 128, 128, "bf16", h0_std=0.5, seed=42)
        d = dev(inp)
        o, hT, ws = g.linear_attn_fwd(d["q"], d["k"], d["v"], d["h0"], d["cu_seqlens"])
        assert g.workspace_status(ws) == 0
        ro, rh = oracle.linear(inp["q"], inp["k"], inp["v"], inp["h0"], inp["cu_seqlens"])
    assert rel(o, ro) <= TOL["bf16"], rel(o, ro)
    assert rel(hT, rh) <= TOL["bf16"], rel(hT, rh)


def test_two_level_scan_without_h0_or_final_state(g, monkeypatch):
    monkeypatch.setenv("GDN_TWO_LEVEL", "3")
    inp = gi.gdn_inputs([900, 130], 4, 128, 128, "bf16", h0_std=0.0, seed=43)
    d = dev(inp)
    o, hT, ws = g.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], None,
                                d["cu_seqlens"], output_final_state=False)
    assert hT is None and g.workspace_status(ws) == 0
    ro, _ = oracle.gdn(inp["q"], inp["k"], inp["v"], inp["log_alpha"], inp["beta"], None,
                       inp["cu_seqlens"])
    assert rel(o, ro) <= TOL["bf16"]


def test_two_level_scan_reports_malformed_seqlens(g, monkeypatch):
    monkeypatch.setenv("GDN_TWO_LEVEL", "4")
    inp = gi.gdn_inputs([64, 64], 4, 128, 128, "bf16", h0_std=0.0, seed=44)
    d = dev(inp)
    cu = torch.tensor([0, 100, 64], dtype=torch.int32, device="cuda")
    _, _, ws = g.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], None, cu)
    assert g.workspace_status(ws) == -4


def test_two_level_scan_forced_timeout_then_recovery(g, monkeypatch):
    """Every bounded wait gives up at once in the scan's runs: the call ends
    with GDN_ERR_TIMEOUT and a barrier site in the caller's workspace, and a
    normal call on the same workspace then matches the oracle."""
    monkeypatch.setenv("GDN_TWO_LEVEL", "3")
    inp = gi.gdn_inputs([500, 257], 4, 128, 128, "bf16", h0_std=0.01, seed=45)
    d = dev(inp)
    args = [d[k] for k in ("q", "k", "v", "log_alpha", "beta", "h0", "cu_seqlens")]
    old = g.set_wait_limit(0)
    try:
        _, _, ws = g.gdn_chunk_fwd(*args)
        assert g.workspace_status(ws) == -9
        assert g.workspace_timeout_site(ws) != 0
    finally:
        g.set_wait_limit(old)
    o, hT, _ = g.gdn_chunk_fwd(*args, workspace=ws)
    assert g.workspace_status(ws) == 0
    ro, rh = ref_gdn(inp)
    assert rel(o, ro) <= TOL["bf16"] and rel(hT, rh) <= TOL["bf16"]


def test_two_level_scan_default_t131072_h4(g, monkeypatch):
    """A 131072-token sequence with 4 heads: the automatic choice cuts it into
    segments (4 chains alone would keep 12 of the SMs busy).  Two heads,
    every token, and all final states against the oracle."""
    monkeypatch.delenv("GDN_TWO_LEVEL", raising=False)
    inp = gi.gdn_inputs([131072], 4, 128, 128, "bf16", h0_std=0.01, seed=0)
    o, hT = run_gdn(g, inp)
    check_chains(inp, o, hT, [(0, 1), (0, 3)], TOL["bf16"])


# ------------------------------------------------------------------ linear-attention variants

@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("normalize", [True, False])
def test_linear_variants_against_oracle(g, causal, normalize):
    """Causal or bidirectional, normalised or not, on ragged packed sequences
    (a one-token and an empty sequence included): every output, K^T V and the
    summed keys against the oracle's quadratic form."""
    lengths = [1, 100, 0, 257, 64, 700]
    inp = gi.linear_inputs(lengths, 4, 128, 128, "bf16", seed=51)
    d = dev(inp)
    o, kv, z, ws = g.linear_attn_variant(d["q"], d["k"], d["v"], d["cu_seqlens"], causal=causal,
                                         normalize=normalize, output_kv=True, output_z=True)
    assert g.workspace_status(ws) == 0
    ro, rkv, rz = oracle.linear_variant(inp["q"], inp["k"], inp["v"], inp["cu_seqlens"], causal=causal,
                                        normalize=normalize)
    assert rel(o, ro) <= TOL["bf16"], rel(o, ro)
    assert rel(kv, rkv) <= TOL["bf16"], rel(kv, rkv)
    assert rel(z, rz) <= TOL["bf16"], rel(z, rz)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("normalize", [True, False])
def test_linear_variants_b2_t4096_h8(g, causal, normalize):
    """The linear-attention workload's shapes (2 x 4096 tokens, H = 8): every
    output against the oracle."""
    inp = gi.linear_inputs([4096, 4096], 8, 128, 128, "bf16", seed=0)
    d = dev(inp)
    o, _, _, ws = g.linear_attn_variant(d["q"], d["k"], d["v"], d["cu_seqlens"], causal=causal,
                                        normalize=normalize)
    assert g.workspace_status(ws) == 0
    ro, _, _ = oracle.linear_variant(inp["q"], inp["k"], inp["v"], inp["cu_seqlens"], causal=causal,
                                     normalize=normalize)
    assert rel(o, ro) <= TOL["bf16"], rel(o, ro)


def test_linear_bidirectional_normalised_t131072_h32(g):
    """One 131072-token sequence, H = 32, bidirectional and normalised: K^T V
    and the summed keys of every head against the oracle's sums, and sampled
    tokens of every head against q_t (K^T V) / (q_t . z) from those sums (the
    reassociation the oracle pins against its quadratic form)."""
    inp = gi.linear_inputs([131072], 32, 128, 128, "bf16", seed=1)
    d = dev(inp)
    o, kv, z, ws = g.linear_attn_variant(d["q"], d["k"], d["v"], None, causal=False, normalize=True,
                                         output_kv=True, output_z=True)
    assert g.workspace_status(ws) == 0
    rkv, rz = oracle.linear_sums(inp["k"], inp["v"])
    assert rel(kv, rkv) <= TOL["bf16"] and rel(z, rz) <= TOL["bf16"]
    ts = torch.randint(0, 131072, (64,), generator=torch.Generator().manual_seed(5))
    qs = inp["q"][ts].double().numpy()  # [64, H, dk]
    ref = np.einsum("thi,hij->thj", qs, rkv[0]) / np.einsum("thi,hi->th", qs, rz[0])[..., None]
    assert rel(o[ts.cuda()], ref) <= TOL["bf16"]


def test_linear_bidirectional_forced_timeout_then_recovery(g):
    inp = gi.linear_inputs([300, 500], 4, 128, 128, "bf16", seed=52)
    d = dev(inp)
    old = g.set_wait_limit(0)
    try:
        _, _, _, ws = g.linear_attn_variant(d["q"], d["k"], d["v"], d["cu_seqlens"], causal=False,
                                            normalize=True)
        assert g.workspace_status(ws) in (0, -9)
    finally:
        g.set_wait_limit(old)
    o, _, _, _ = g.linear_attn_variant(d["q"], d["k"], d["v"], d["cu_seqlens"], causal=False,
                                       normalize=True, workspace=ws)
    assert g.workspace_status(ws) == 0
    ro, _, _ = oracle.linear_variant(inp["q"], inp["k"], inp["v"], inp["cu_seqlens"], causal=False,
                                     normalize=True)
    assert rel(o, ro) <= TOL["bf16"]


# ------------------------------------------------------------------ the plan at the one-warp boundary

@pytest.mark.parametrize("n_seqs", [32, 33])
def test_plan_boundary_gdn_and_linear(g, monkeypatch, n_seqs):
    """32 sequences take the plan's one-warp path (one lane copies two offsets),
    33 the block-wide one: every output and final state of GDN and of the
    grouped linear attention against the oracle (ragged lengths, an empty
    sequence, a one-token one)."""
    monkeypatch.delenv("GDN_LINEAR_PATH", raising=False)
    gen = torch.Generator().manual_seed(70 + n_seqs)
    lengths = [int(x) for x in torch.randint(1, 300, (n_seqs,), generator=gen)]
    lengths[3], lengths[7] = 0, 1
    inp = gi.gdn_inputs(lengths, 2, 128, 128, "bf16", h0_std=0.01, seed=71)
    o, hT = run_gdn(g, inp)
    ro, rh = ref_gdn(inp)
    assert rel(o, ro) <= TOL["bf16"] and rel(hT, rh) <= TOL["bf16"]
    lin = gi.linear_inputs(lengths, 2, 128, 128, "bf16", h0_std=0.1, seed=72)
    d = dev(lin)
    o2, h2, ws = g.linear_attn_fwd(d["q"], d["k"], d["v"], d["h0"], d["cu_seqlens"])
    assert g.workspace_status(ws) == 0
    ro2, rh2 = oracle.linear(lin["q"], lin["k"], lin["v"], lin["h0"], lin["cu_seqlens"])
    assert rel(o2, ro2) <= TOL["bf16"] and rel(h2, rh2) <= TOL["bf16"]


# ------------------------------------------------------------------ causal linear attention, grouped

@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("lengths,H,h0_std", [([1, 100, 0, 257, 64, 700], 4, 0.5), ([3000, 1500], 8, 0.0),
                                              ([64, 65, 63, 128, 1], 4, 0.1)])
def test_linear_grouped_against_oracle(g, monkeypatch, lengths, H, h0_std, fused):
    """Causal linear attention through groups of chunks (the default path of
    linear_attn_fwd for bf16, d = 128), in one cooperative launch (fused) and
    as separate sum, prefix and apply kernels: ragged sequences, several
    groups per sequence, partial and empty chunks, with and without h0; every
    output and every final state against the oracle's recurrence."""
    monkeypatch.delenv("GDN_LINEAR_PATH", raising=False)
    monkeypatch.delenv("GDN_PREFILL_PAIR", raising=False)
    monkeypatch.delenv("GDN_TWO_LEVEL", raising=False)
    monkeypatch.setenv("GDN_LINEAR_GROUPED_FORM", "fused" if fused else "unfused")
    inp = gi.linear_inputs(lengths, H, 128, 128, "bf16", h0_std=h0_std, seed=61)
    d = dev(inp)
    o, hT, ws = g.linear_attn_fwd(d["q"], d["k"], d["v"], d["h0"], d["cu_seqlens"])
    assert g.workspace_status(ws) == 0
    ro, rh = oracle.linear(inp["q"], inp["k"], inp["v"], inp["h0"], inp["cu_seqlens"])
    assert rel(o, ro) <= TOL["bf16"], rel(o, ro)
    assert rel(hT, rh) <= TOL["bf16"], rel(hT, rh)


def test_linear_grouped_many_sequences(g, monkeypatch):
    """More (sequence, head) pairs than SMs (44 sequences x 4 heads), so the
    group size comes from the total, not from the one-wave search: every
    output and final state, normalised and not, against the oracle."""
    monkeypatch.delenv("GDN_LINEAR_PATH", raising=False)
    lengths = [int(x) for x in torch.randint(1, 700, (44,), generator=torch.Generator().manual_seed(64))]
    inp = gi.linear_inputs(lengths, 4, 128, 128, "bf16", h0_std=0.1, seed=64)
    d = dev(inp)
    o, hT, ws = g.linear_attn_fwd(d["q"], d["k"], d["v"], d["h0"], d["cu_seqlens"])
    assert g.workspace_status(ws) == 0
    ro, rh = oracle.linear(inp["q"], inp["k"], inp["v"], inp["h0"], inp["cu_seqlens"])
    assert rel(o, ro) <= TOL["bf16"] and rel(hT, rh) <= TOL["bf16"]
    on, _, _, ws = g.linear_attn_variant(d["q"], d["k"], d["v"], d["cu_seqlens"], causal=True, normalize=True)
    assert g.workspace_status(ws) == 0
    rn, _, _ = oracle.linear_variant(inp["q"], inp["k"], inp["v"], inp["cu_seqlens"], causal=True, normalize=True)
    assert rel(on, rn) <= TOL["bf16"], rel(on, rn)


def test_linear_grouped_t131072_h32(g, monkeypatch):
    """One 131072-token sequence, H = 32, through groups: sampled heads, every
    token, and all final states against the oracle."""
    monkeypatch.delenv("GDN_LINEAR_PATH", raising=False)
    inp = gi.linear_inputs([131072], 32, 128, 128, "bf16", h0_std=0.1, seed=62)
    d = dev(inp)
    o, hT, ws = g.linear_attn_fwd(d["q"], d["k"], d["v"], d["h0"], d["cu_seqlens"])
    assert g.workspace_status(ws) == 0
    hs = [0, 19]
    ro, rh = oracle.linear(inp["q"][:, hs], inp["k"][:, hs], inp["v"][:, hs], inp["h0"][:, hs])
    assert rel(o[:, hs], ro) <= TOL["bf16"] and rel(hT[:, hs], rh) <= TOL["bf16"]
    rkv, _ = oracle.linear_sums(inp["k"], inp["v"])
    assert rel(hT, inp["h0"].double().numpy() + rkv) <= TOL["bf16"]


@pytest.mark.parametrize("fused", [True, False])
def test_linear_grouped_forced_timeout_then_recovery(g, monkeypatch, fused):
    monkeypatch.delenv("GDN_LINEAR_PATH", raising=False)
    monkeypatch.setenv("GDN_LINEAR_GROUPED_FORM", "fused" if fused else "unfused")
    inp = gi.linear_inputs([700, 300], 4, 128, 128, "bf16", h0_std=0.1, seed=63)
    d = dev(inp)
    args = [d[k] for k in ("q", "k", "v", "h0", "cu_seqlens")]
    old = g.set_wait_limit(0)
    try:
        _, _, ws = g.linear_attn_fwd(*args)
        assert g.workspace_status(ws) in (0, -9)
    finally:
        g.set_wait_limit(old)
    o, hT, _ = g.linear_attn_fwd(*args, workspace=ws)
    assert g.workspace_status(ws) == 0
    ro, rh = oracle.linear(inp["q"], inp["k"], inp["v"], inp["h0"], inp["cu_seqlens"])
    assert rel(o, ro) <= TOL["bf16"] and rel(hT, rh) <= TOL["bf16"]


# ------------------------------------------------------------------ failure detection

@pytest.mark.parametrize("kernel", KERNELS)
def test_forced_wait_timeout_then_recovery(g, monkeypatch, kernel):
    """With the wait bound at 0 every bounded device wait gives up at once:
    the call must end (no hang), report GDN_ERR_TIMEOUT and the barrier it
    gave up on in the workspace, and leave the context usable; a normal call
    on the same workspace right after matches the oracle."""
    use_kernel(monkeypatch, kernel)
    inp = gi.gdn_inputs([300, 77, 129], 4, 128, 128, "bf16", h0_std=0.01, seed=17)
    d = dev(inp)
    args = [d[k] for k in ("q", "k", "v", "log_alpha", "beta", "h0", "cu_seqlens")]
    old = g.set_wait_limit(0)
    try:
        _, _, ws = g.gdn_chunk_fwd(*args)
        assert g.workspace_status(ws) == -9  # GDN_ERR_TIMEOUT
        assert g.workspace_timeout_site(ws) != 0
    finally:
        assert g.set_wait_limit(old) == 0
    o, hT, ws2 = g.gdn_chunk_fwd(*args, workspace=ws)
    assert ws2 is ws and g.workspace_status(ws) == 0 and g.workspace_timeout_site(ws) == 0
    ro, rh = ref_gdn(inp)
    assert rel(o, ro) <= TOL["bf16"] and rel(hT, rh) <= TOL["bf16"]


# ------------------------------------------------------------------ decode

def test_decode_b128_h32(g):
    """Decode: 128 sequences x 32 heads, d = 128, fp32 state in place.
    The full state after 16 steps, and 8 sampled chains over 1024 steps."""
    B, H, D = 128, 32, 128
    state0 = gi.decode_state(B, H, D, D, seed=0)
    state = state0.cuda()
    chains = [(0, 0), (5, 31), (17, 3), (64, 16), (99, 8), (127, 31), (33, 12), (90, 25)]
    ref_state = {c: state0[c[0], c[1]].double().numpy() for c in chains}
    full_ref = state0.double().numpy()
    steps = 1024
    worst_o = 0.0
    for step in range(steps):
        inp = gi.decode_step_inputs(B, H, D, D, step, seed=0)
        d = dev(inp)
        o = g.gdn_recurrent_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], state)
        o_cpu = o.double().cpu().numpy()
        if step < 16:
            ro, full_ref = oracle.decode_step(inp["q"], inp["k"], inp["v"], inp["log_alpha"],
                                              inp["beta"], full_ref)
            assert rel(o_cpu, ro) <= TOL["bf16"], (step, rel(o_cpu, ro))
            if step == 15:
                assert rel(state, full_ref) <= TOL["bf16"]
        for (b, h) in chains:
            ro, st = oracle.decode_step(inp["q"][b:b + 1, h:h + 1], inp["k"][b:b + 1, h:h + 1],
                                        inp["v"][b:b + 1, h:h + 1], inp["log_alpha"][b:b + 1, h:h + 1],
                                        inp["beta"][b:b + 1, h:h + 1],
                                        ref_state[(b, h)][None, None])
            ref_state[(b, h)] = st[0, 0]
            worst_o = max(worst_o, float(np.max(np.abs(o_cpu[b, h] - ro[0, 0]))) /
                          max(float(np.max(np.abs(ro[0, 0]))), 1e-30))
    assert worst_o <= TOL["bf16"], worst_o
    got = np.stack([state[b, h].double().cpu().numpy() for b, h in chains])
    ref = np.stack([ref_state[c] for c in chains])
    assert rel(got, ref) <= TOL["bf16"], rel(got, ref)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64)])
def test_decode_small_heads(g, dk, dv):
    B, H = 3, 5
    state0 = gi.decode_state(B, H, dk, dv, seed=1)
    state = state0.cuda()
    ref = state0.double().numpy()
    for step in range(5):
        inp = gi.decode_step_inputs(B, H, dk, dv, step, seed=1)
        d = dev(inp)
        o = g.gdn_recurrent_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], state)
        ro, ref = oracle.decode_step(inp["q"], inp["k"], inp["v"], inp["log_alpha"], inp["beta"], ref)
        assert rel(o, ro) <= TOL["bf16"]
    assert rel(state, ref) <= TOL["bf16"]


# ------------------------------------------------------------------ edge cases

def test_single_sequence_without_cu_seqlens(g):
    inp = gi.gdn_inputs([333], 2, 128, 128, "bf16", h0_std=0.01, seed=6)
    d = dev(inp)
    o, hT, ws = g.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["h0"], None)
    assert g.workspace_status(ws) == 0
    ro, rh = ref_gdn(inp)
    assert rel(o, ro) <= TOL["bf16"] and rel(hT, rh) <= TOL["bf16"]


@pytest.mark.parametrize("lengths", [[1], [0, 1, 0], [64], [65], [0, 0]])
def test_tiny_and_empty(g, lengths):
    inp = gi.gdn_inputs(lengths, 2, 128, 128, "bf16", h0_std=0.01, seed=7)
    o, hT = run_gdn(g, inp)
    ro, rh = ref_gdn(inp)
    if sum(lengths):
        assert rel(o, ro) <= TOL["bf16"]
    assert rel(hT, rh) <= TOL["bf16"]
    for s, L in enumerate(lengths):  # zero-length sequences return h0 exactly
        if L == 0:
            assert torch.equal(hT[s].cpu(), inp["h0"][s])


def test_no_h0_and_no_final_state(g):
    inp = gi.gdn_inputs([100, 50], 2, 128, 128, "bf16", h0_std=0.0, seed=8)
    d = dev(inp)
    o, hT, ws = g.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], None,
                                d["cu_seqlens"], output_final_state=False)
    assert hT is None and g.workspace_status(ws) == 0
    ro, _ = ref_gdn(inp)
    assert rel(o, ro) <= TOL["bf16"]


def test_state_chaining_across_calls(g):
    """h_T of a first call used as h0 of a second equals one call."""
    inp = gi.gdn_inputs([1000], 2, 128, 128, "bf16", h0_std=0.01, seed=9)
    d = dev(inp)
    o, hT = run_gdn(g, inp)
    cut = 390
    o1, h1, _ = g.gdn_chunk_fwd(d["q"][:cut].contiguous(), d["k"][:cut].contiguous(),
                                d["v"][:cut].contiguous(), d["log_alpha"][:cut].contiguous(),
                                d["beta"][:cut].contiguous(), d["h0"], None)
    o2, h2, _ = g.gdn_chunk_fwd(d["q"][cut:].contiguous(), d["k"][cut:].contiguous(),
                                d["v"][cut:].contiguous(), d["log_alpha"][cut:].contiguous(),
                                d["beta"][cut:].contiguous(), h1, None)
    both = torch.cat([o1, o2]).double().cpu().numpy()
    assert rel(o, both) <= TOL["bf16"]
    assert rel(hT, h2.double().cpu().numpy()) <= TOL["bf16"]


def test_outputs_written_only_in_bounds(g):
    """Canary rows after o and h_T stay untouched (partial last chunks)."""
    lengths = [70, 3, 129]
    inp = gi.gdn_inputs(lengths, 2, 128, 128, "bf16", h0_std=0.01, seed=10)
    d = dev(inp)
    T = sum(lengths)
    o_buf = torch.full((T + 64, 2, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    h_buf = torch.full((len(lengths) + 1, 2, 128, 128), 7.0, device="cuda")
    o, hT, ws = g.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["h0"],
                                d["cu_seqlens"], o=o_buf[:T], h_T=h_buf[:len(lengths)])
    assert g.workspace_status(ws) == 0
    assert bool((o_buf[T:] == 7.0).all()) and bool((h_buf[len(lengths):] == 7.0).all())
    ro, rh = ref_gdn(inp)
    assert rel(o, ro) <= TOL["bf16"] and rel(hT, rh) <= TOL["bf16"]


def test_malformed_cu_seqlens_reported_on_device(g):
    inp = gi.gdn_inputs([64, 64], 1, 128, 128, "bf16", h0_std=0.0, seed=11)
    d = dev(inp)
    for bad in ([0, 100, 64, 128], [5, 64, 128], [0, 64, 127]):
        cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
        n = len(bad) - 1
        o = torch.zeros(128, 1, 128, dtype=torch.bfloat16, device="cuda")
        hT = torch.zeros(n, 1, 128, 128, device="cuda")
        _, _, ws = g.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], None, cu,
                                   o=o, h_T=hT)
        assert g.workspace_status(ws) == -4
        _, _, ws = g.gdn_chunk_fwd_staged(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], None,
                                          cu, o=o, h_T=hT)
        assert g.workspace_status(ws) == -4


def test_workspace_reused_across_calls(g):
    a = gi.gdn_inputs([500, 20], 2, 128, 128, "bf16", h0_std=0.01, seed=12)
    b = gi.gdn_inputs([80], 2, 128, 128, "bf16", h0_std=0.01, seed=13)
    _, _, ws = g.gdn_chunk_fwd(*[dev(a)[k] for k in ("q", "k", "v", "log_alpha", "beta", "h0", "cu_seqlens")])
    db = dev(b)
    o, hT, ws2 = g.gdn_chunk_fwd(db["q"], db["k"], db["v"], db["log_alpha"], db["beta"], db["h0"],
                                 db["cu_seqlens"], workspace=ws)
    assert ws2 is ws and g.workspace_status(ws) == 0
    ro, rh = ref_gdn(b)
    assert rel(o, ro) <= TOL["bf16"] and rel(hT, rh) <= TOL["bf16"]
