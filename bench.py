"""Benchmark: GDN long prefill on B300, tokens/s and fraction of roofline.

Workload: 4 packed sequences with seeded lengths summing to T = 131072 tokens,
H = 32 heads, dk = dv = 128, bf16 q/k/v/o, fp32 gates and states, chunk 64
(one gdn_chunk_fwd call per step).  Inputs are seeded synthetic tensors far
larger than L2 (4.35 GB), so no L2 flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --workload {gdn_t32768_h16, gdn_t131072_h32_single, gdn_t65536_h8, linear_b2_t4096_h8,
                              decode_b128_h32, gdn_varlen_t131072_h32_block_adjacent, gdn_t131072_h4,
                              linear_bidir_norm_b2_t4096_h8, linear_causal_norm_b2_t4096_h8,
                              linear_bidir_norm_t131072_h32, linear_causal_norm_t131072_h32,
                              linear_bidir_norm_t32768_h32 (any _t<T>_h<H>)}
                                                   (the other workloads, one GPU)

One JSON line is printed by rank 0.  Under torchrun each rank runs the same
per-GPU workload on its own GPU (weak scaling, no collective on the data
path); `value` is the total tokens of all ranks over the slowest rank's time.
`--impl reference` times the fp64 CPU oracle instead, on a bounded sample.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gdn_inputs as gi  # noqa: E402

KERNEL_SRC = {"fused_single_sm": "fused_tc.cu", "fused_pair": "fused_cluster.cu"}


def kernel_name(fused, units=None):
    """Which prefill kernel gdn_chunk_fwd runs (the library's own dispatch rule:
    the 2-SM cluster kernel unless GDN_PREFILL_PAIR=0)."""
    if not fused:
        return "staged"
    return "fused_single_sm" if os.environ.get("GDN_PREFILL_PAIR", "") == "0" else "fused_pair"


def linear_grouped():
    """Whether linear_attn_fwd (bf16, d = 128) takes the grouped causal path
    (the library's own rule: yes unless GDN_LINEAR_PATH=cluster,
    GDN_PREFILL_PAIR=0 or GDN_TWO_LEVEL picks the fused kernels)."""
    if os.environ.get("GDN_LINEAR_PATH", "") == "cluster" or os.environ.get("GDN_PREFILL_PAIR", "") == "0":
        return False
    return os.environ.get("GDN_TWO_LEVEL", "") == ""


def source_digest(kernel):
    import hashlib
    path = os.path.join(ROOT, "gated_deltanet_sequence_prefill_b300", "csrc", KERNEL_SRC.get(kernel, ""))
    if not os.path.isfile(path):
        return None
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per call from the committed ncu summary, or None when there is
    none for this kernel or the kernel source changed since it was taken."""
    prof = os.path.join(ROOT, "profiles", "traffic_gdn_varlen_t131072_h32.json")
    if not os.path.exists(prof):
        return None
    with open(prof) as f:
        t = json.load(f)
    if t.get("kernel") != kernel or t.get("source_sha256_16") != source_digest(kernel):
        return None
    return t.get("bytes_per_call")

METRIC = "GDN prefill tokens/s at H=32,d=128,T=128K bf16; % of roofline (1×B300)"
T_TOTAL, H, D = 131072, 32, 128
LENGTHS = gi.varlen_lengths(T_TOTAL, 4, 0)
WORKLOAD = "gdn_varlen_t131072_h32_d128"


def alg_bytes():
    """Algorithmic bytes of one call: q, k, v in and o out (bf16), the two fp32
    gates, h0 in and h_T out (fp32)."""
    n = len(LENGTHS)
    return (4 * T_TOTAL * H * D * 2) + (2 * T_TOTAL * H * 4) + (2 * n * H * D * D * 4)


def alg_flops():
    """Algorithmic flops per token per head at chunk 64, d = 128: three state
    contractions (w h, q h, k~^T v_new: 6 d^2), the causal halves of the five
    chunk-local products (5 C d) and the triangular solve (C^2 / 3)."""
    C = 64
    return T_TOTAL * H * (6 * D * D + 5 * C * D + C * C / 3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]), src="measured")
    return dict(hbm=6400.0, bf16=1800.0, src="fallback")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.time()  # make sure sampling runs before the timed region starts
            while not self.lines and time.time() - t0 < 5.0:
                time.sleep(0.02)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        time.sleep(0.25)  # at least a couple of samples from the end of the timed region
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(budget_s=15.0):
    """The fp64 oracle (as it stands) on a bounded sample of the workload: the
    first S tokens of each of the 4 sequences, all 32 heads; S is grown until
    one run takes a few seconds, then the rate is measured on one larger run."""
    import oracle
    inp = gi.gdn_inputs(LENGTHS, H, D, D, "bf16", h0_std=0.01, seed=0)
    cu = inp["cu_seqlens"].tolist()

    def sample(S):
        idx = []
        lens = []
        for s in range(len(LENGTHS)):
            n = min(S, LENGTHS[s])
            idx.extend(range(cu[s], cu[s] + n))
            lens.append(n)
        sl = lambda x: x[idx].contiguous()
        cus = [0]
        for n in lens:
            cus.append(cus[-1] + n)
        return (sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["log_alpha"]), sl(inp["beta"]),
                inp["h0"], cus), sum(lens)

    S, elapsed, tokens = 16, 0.0, 0
    while True:
        args, tokens = sample(S)
        t0 = time.perf_counter()
        oracle.gdn(*args)
        elapsed = time.perf_counter() - t0
        if elapsed > budget_s / 4 or S >= max(LENGTHS):
            break
        S = min(max(LENGTHS), int(S * max(2.0, (budget_s / 2) / max(elapsed, 1e-3))))
    return {"value": tokens / elapsed, "unit": "tokens/s", "cores": oracle.num_threads(),
            "host_cpus": os.cpu_count(), "kind": "oracle", "seconds": elapsed,
            "sample": "fp64 token recurrence on the first %d tokens of each of the 4 sequences, "
                      "all 32 heads (%d tokens x 32 heads)" % (S, tokens)}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    inp = gi.gdn_inputs(LENGTHS, H, D, D, "bf16", h0_std=0.01, seed=0)
    cu = inp["cu_seqlens"].tolist()
    S = 256  # tokens of each sequence per step: a bounded sample of the workload
    idx = [t for s in range(4) for t in range(cu[s], cu[s] + S)]
    sl = lambda x: x[idx].contiguous()
    step_args = (sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["log_alpha"]), sl(inp["beta"]),
                 inp["h0"], [0, S, 2 * S, 3 * S, 4 * S])
    for _ in range(args.warmup):
        oracle.gdn(*step_args)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gdn(*step_args)
    dt = (time.perf_counter() - t0) / args.steps
    tokens = 4 * S
    value = tokens / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": T_TOTAL, "H": H, "dk": D, "dv": D,
                   "seq_lens": LENGTHS, "chunk": 64},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": "first %d tokens of each of the 4 sequences, all 32 heads, "
                                   "per step" % S},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def max_over_ranks(x, dist=None, device=None):
    """The slowest rank's figure.  Every rank runs the same per-GPU workload
    (weak scaling, no collective on the data path), so the job takes as long as
    its slowest rank; with one process this is x itself."""
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, tokens_per_rank, ms_per_step):
    """Whole-job throughput: the tokens all ranks processed over the slowest
    rank's time."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


def run_ours(args, rank, world, local_rank):
    import torch
    import gated_deltanet_sequence_prefill_b300 as g
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    inp = gi.gdn_inputs(LENGTHS, H, D, D, "bf16", h0_std=0.01, seed=0)
    dv = {k: v.cuda() for k, v in inp.items()}
    T = T_TOTAL
    n = len(LENGTHS)
    o = torch.empty(T, H, D, dtype=torch.bfloat16, device="cuda")
    hT = torch.empty(n, H, D, D, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(g.chunk_fwd_workspace_size(T, H, D, D, n), 256), dtype=torch.uint8,
                     device="cuda")
    fused = g.chunk_fwd_workspace_size(T, H, D, D, n) < g.staged_workspace_size(T, H, D, D, n)
    launches_per_call = 2 if fused else 4
    stream = torch.cuda.current_stream()

    def call():
        g.gdn_chunk_fwd(dv["q"], dv["k"], dv["v"], dv["log_alpha"], dv["beta"], dv["h0"],
                        dv["cu_seqlens"], o=o, h_T=hT, workspace=ws)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    assert g.workspace_status(ws) == 0

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        t_end.record(stream)
        barrier()
    total_ms = t_start.elapsed_time(t_end)
    per_call = [a.elapsed_time(b) for a, b in ev]
    status = g.workspace_status(ws)
    if status != 0:
        raise RuntimeError("device status %d" % status)

    ms_per_step = max_over_ranks(total_ms / args.steps, dist, "cuda")
    value = job_tokens_per_s(world, T, ms_per_step)

    # end to end through the same public call, from and to pinned host memory: every
    # step uploads its inputs, runs the call and reads o and h_T back.  Uploads and
    # read-backs go on their own streams (the link is full duplex), with the device
    # inputs double-buffered, so step i + 1's upload overlaps step i's call and read-back.
    host = {k: v.pin_memory() for k, v in inp.items()}
    o_host = torch.empty(T, H, D, dtype=torch.bfloat16).pin_memory()
    h_host = torch.empty(n, H, D, D, dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = o_host.numel() * 2 + h_host.numel() * 4
    e2e_steps = max(2, min(args.steps, 5))
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    dbuf = [{k: torch.empty_like(v, device="cuda") for k, v in host.items()} for _ in range(2)]
    obuf = [torch.empty(T, H, D, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    hbuf = [torch.empty(n, H, D, D, dtype=torch.float32, device="cuda") for _ in range(2)]

    def e2e_run(steps):
        done = [None, None]  # read-back of the step that last used each buffer pair
        for i in range(steps):
            b = i % 2
            if done[b] is not None:
                up.wait_event(done[b])  # that step's call has consumed these inputs
            with torch.cuda.stream(up):
                for k, v in host.items():
                    dbuf[b][k].copy_(v, non_blocking=True)
                landed = torch.cuda.Event()
                landed.record(up)
            stream.wait_event(landed)
            dd = dbuf[b]
            g.gdn_chunk_fwd(dd["q"], dd["k"], dd["v"], dd["log_alpha"], dd["beta"], dd["h0"], dd["cu_seqlens"],
                            o=obuf[b], h_T=hbuf[b], workspace=ws, stream=stream)
            ran = torch.cuda.Event()
            ran.record(stream)
            down.wait_event(ran)
            with torch.cuda.stream(down):
                o_host.copy_(obuf[b], non_blocking=True)
                h_host.copy_(hbuf[b], non_blocking=True)
                done[b] = torch.cuda.Event()
                done[b].record(down)

    e2e_run(2)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_stream(stream)
    e2e_run(e2e_steps)
    stream.wait_stream(down)
    e1.record(stream)
    barrier()
    e2e_value = job_tokens_per_s(world, T, max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, "cuda"))

    if rank == 0:
        pk = peaks()
        kern_ms = statistics.median(per_call)
        achieved = alg_bytes() / (kern_ms / 1e3) / 1e9
        traffic = recorded_traffic(kernel_name(fused, n * H))
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; q,k L2-normalised N(0,1), v N(0,1), "
                    "log_alpha=-softplus(N)*0.1, beta=sigmoid(N), h0 N(0,0.01))",
            "config": {"workload": WORKLOAD, "T": T, "H": H, "dk": D, "dv": D, "seq_lens": LENGTHS,
                       "chunk": 64, "path": kernel_name(fused, n * H),
                       "l2": "inputs larger than L2 (%.2f GB per call), no flush" % (alg_bytes() / 1e9)},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
                         "frac": achieved / pk["hbm"], "traffic": traffic,
                         "peak_source": pk["src"],
                         "kernel_ms": kern_ms,
                         "roofline_ms": 1e3 * max(alg_bytes() / (pk["hbm"] * 1e9),
                                                  alg_flops() / (pk["bf16"] * 1e12)),
                         "note": "algorithmic bytes / median duration of one gdn_chunk_fwd call "
                                 "(plan kernel + prefill kernels), CUDA events on its stream"},
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "note": "gdn_chunk_fwd per step with its inputs uploaded from pinned host memory and o, "
                            "h_T read back; uploads and read-backs on their own streams, overlapping the "
                            "neighbouring steps"},
            "gpu_launches": launches_per_call * args.steps,
            "clocks": clk.summary(),
        }
        line["roofline"]["frac_of_time_roofline"] = line["roofline"]["roofline_ms"] / kern_ms
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def run_workload(args):
    """Time one of the other workloads on one GPU (same timing rules)."""
    import torch
    import gated_deltanet_sequence_prefill_b300 as g
    torch.cuda.set_device(0)
    pk = peaks()
    stream = torch.cuda.current_stream()
    flush = None
    name = args.workload
    if name == "decode_b128_h32":
        B, Hh, Dd, steps = 128, 32, 128, 1024
        gen = torch.Generator(device="cuda")
        gen.manual_seed(0)
        state = (torch.randn(B, Hh, Dd, Dd, generator=gen, device="cuda") * 0.01).float()

        def step_inputs():
            q = torch.randn(B, Hh, Dd, generator=gen, device="cuda")
            k = torch.randn(B, Hh, Dd, generator=gen, device="cuda")
            q = (q / q.norm(dim=-1, keepdim=True)).bfloat16()
            k = (k / k.norm(dim=-1, keepdim=True)).bfloat16()
            v = torch.randn(B, Hh, Dd, generator=gen, device="cuda").bfloat16()
            la = (-torch.nn.functional.softplus(torch.randn(B, Hh, generator=gen, device="cuda")) * 0.1).bfloat16()
            be = torch.sigmoid(torch.randn(B, Hh, generator=gen, device="cuda")).bfloat16()
            return q, k, v, la, be
        inputs = [step_inputs() for _ in range(steps)]
        o = torch.empty(B, Hh, Dd, dtype=torch.bfloat16, device="cuda")

        def run():
            for q, k, v, la, be in inputs:
                g.gdn_recurrent_step(q, k, v, la, be, state, o=o)
        units, unit = B * steps, "tokens/s"
        bytes_per_call = steps * (2 * B * Hh * Dd * Dd * 4 + 4 * B * Hh * Dd * 2 + 2 * B * Hh * 2)
        launches = steps
        cfg = {"workload": name, "B": B, "H": Hh, "dk": Dd, "dv": Dd, "steps_per_call": steps,
               "l2": "state 537 MB per step, larger than L2, no flush"}
    else:
        if name == "linear_b2_t4096_h8":
            lengths, Hh, kind = [4096, 4096], 8, "linear"
            inp = gi.linear_inputs(lengths, Hh, D, D, "bf16", seed=0)
            flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        elif name == "gdn_t32768_h16":
            lengths, Hh, kind = [32768], 16, "gdn"
            inp = gi.gdn_inputs(lengths, Hh, D, D, "bf16", h0_std=0.01, seed=0)
        elif name == "gdn_t131072_h32_single":
            lengths, Hh, kind = [131072], 32, "gdn"
            inp = gi.gdn_inputs(lengths, Hh, D, D, "bf16", h0_std=0.01, seed=0)
        elif name == "gdn_t65536_h8":  # the small case the ncu summaries capture
            lengths, Hh, kind = [65536], 8, "gdn"
            inp = gi.gdn_inputs(lengths, Hh, D, D, "bf16", h0_std=0.01, seed=0)
        elif name == "gdn_t16384_h64":  # many concurrent units, small enough for ncu sections
            lengths, Hh, kind = [16384], 64, "gdn"
            inp = gi.gdn_inputs(lengths, Hh, D, D, "bf16", h0_std=0.01, seed=0)
        elif name == "gdn_t16384_h4":  # the same length with few units
            lengths, Hh, kind = [16384], 4, "gdn"
            inp = gi.gdn_inputs(lengths, Hh, D, D, "bf16", h0_std=0.01, seed=0)
        elif name.startswith("linear_bidir_norm_") or name.startswith("linear_causal_norm_"):
            # linear-attention variants: causal or bidirectional, normalised
            if name.endswith("b2_t4096_h8"):
                lengths, Hh = [4096, 4096], 8
            else:  # ..._t<T>_h<H>: one sequence
                tt, hh = name.rsplit("_", 2)[-2:]
                lengths, Hh = [int(tt[1:])], int(hh[1:])
            kind = "bidir_norm" if "bidir" in name else "causal_norm"
            inp = gi.linear_inputs(lengths, Hh, D, D, "bf16", seed=0)
            if Hh == 8:
                flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        elif name == "gdn_t131072_h4":  # one long sequence, few heads: the two-level state scan
            lengths, Hh, kind = [131072], 4, "gdn"
            inp = gi.gdn_inputs(lengths, Hh, D, D, "bf16", h0_std=0.01, seed=0)
        elif name == "gdn_varlen_t131072_h32_block_adjacent":  # the headline with the approximate solver
            lengths, Hh, kind = LENGTHS, H, "gdn_block_adjacent"
            inp = gi.gdn_inputs(lengths, Hh, D, D, "bf16", h0_std=0.01, seed=0)
        else:
            raise SystemExit("unknown workload " + name)
        d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
        Tt, nn = sum(lengths), len(lengths)
        o = torch.empty(Tt, Hh, D, dtype=torch.bfloat16, device="cuda")
        hT = torch.empty(nn, Hh, D, D, dtype=torch.float32, device="cuda")
        gdn_kind = kind.startswith("gdn")
        wsz = g.chunk_fwd_workspace_size(Tt, Hh, D, D, nn, delta_rule=gdn_kind)
        ws = torch.empty(max(wsz, 256), dtype=torch.uint8, device="cuda")
        if kind in ("bidir_norm", "causal_norm"):
            causal = kind == "causal_norm"
            ws = None

            def run():
                nonlocal ws
                _, _, _, ws = g.linear_attn_variant(d["q"], d["k"], d["v"], d["cu_seqlens"], causal=causal,
                                                    normalize=True, o=o, workspace=ws)
        elif gdn_kind:
            band = kind == "gdn_block_adjacent"

            def run():
                g.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["h0"],
                                d["cu_seqlens"], o=o, h_T=hT, workspace=ws, block_adjacent=band)
        else:
            def run():
                g.linear_attn_fwd(d["q"], d["k"], d["v"], d["h0"], d["cu_seqlens"], o=o, h_T=hT,
                                  workspace=ws)
        units, unit = Tt, "tokens/s"
        bytes_per_call = 4 * Tt * Hh * D * 2 + (2 * Tt * Hh * 4 if gdn_kind else 0) + \
            (2 if gdn_kind else 1) * nn * Hh * D * D * 4
        segs = g.two_level_segments(Tt, Hh, nn, delta_rule=gdn_kind)
        launches = 2 if segs < 2 else (7 if gdn_kind else 6)
        path = kernel_name(True, nn * Hh)
        if kind == "bidir_norm":  # plan, K^T V reduction, apply
            bytes_per_call, launches, segs, path = 4 * Tt * Hh * D * 2, 3, 1, "linear_bidirectional"
        elif kind == "causal_norm" or (kind == "linear" and linear_grouped()):
            # the plan (with the group plan), then one cooperative launch (sums, prefix,
            # apply) for small problems, else half-group K^T V sums, prefix over the
            # groups, group apply
            sms = torch.cuda.get_device_properties(0).multi_processor_count
            form = os.environ.get("GDN_LINEAR_GROUPED_FORM", "")
            fused = Hh * nn <= sms and (form == "fused" or (form != "unfused" and (Tt // 64 + nn) * Hh <= 40 * sms))
            launches, segs = (2 if fused else 4), 1
            path = "linear_grouped_fused" if fused else "linear_grouped"
            if kind == "causal_norm":
                bytes_per_call = 4 * Tt * Hh * D * 2
        cfg = {"workload": name, "T": Tt, "H": Hh, "dk": D, "dv": D, "seq_lens": lengths,
               "two_level_segments": segs,
               "chunk": 64, "path": path, "l2": ("L2 flushed (256 MB write) between timed calls"
                                   if flush is not None else "inputs larger than L2, no flush")}
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    # Each timed step replays a CUDA graph of the same library call (its kernels and
    # arguments, captured once), so that the host's per-call work (argument checks,
    # tensor-map encoding, launches) does not show as idle device time inside the
    # call; the steps are enqueued back to back and timed by events around each.
    graph = None
    if not args.direct:
        try:
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                run()
            torch.cuda.synchronize()
            gr.replay()
            torch.cuda.synchronize()
            graph = gr
        except Exception as ex:  # a path that cannot be captured is timed by direct calls
            cfg["graph_capture_error"] = str(ex)[:200]
    cfg["launch"] = "cuda_graph" if graph is not None else "direct"
    step = graph.replay if graph is not None else run
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(0) as clk:
        for i in range(args.steps):
            if flush is not None:
                flush.fill_(1)
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in ev]
    ws_used = locals().get("ws")
    if isinstance(ws_used, torch.Tensor) and g.workspace_status(ws_used) != 0:
        raise RuntimeError("device status %d" % g.workspace_status(ws_used))
    ms = statistics.median(times)
    achieved = bytes_per_call / (ms / 1e3) / 1e9
    if name.endswith("_block_adjacent"):
        # how far the approximate solve lands from the exact one on these inputs
        o_exact, h_exact, _ = g.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                              d["h0"], d["cu_seqlens"])
        rel = lambda x, y: float((x.double() - y.double()).abs().max() / y.double().abs().max())
        cfg["rel_dev_from_exact_solve"] = {"o": rel(o, o_exact), "h_T": rel(hT, h_exact)}
    line = {"metric": name + " throughput", "value": units / (ms / 1e3), "unit": unit, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic (seeded)", "config": cfg,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
                         "frac": achieved / pk["hbm"], "traffic": None, "peak_source": pk["src"],
                         "alg_bytes_per_call": bytes_per_call},
            "gpu_launches": launches * args.steps, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--direct", action="store_true",
                    help="time --workload runs by direct calls instead of a CUDA graph of the call")
    args = ap.parse_args()
    if args.workload:
        run_workload(args)
        return
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
