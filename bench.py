"""Benchmark of the KDA hot path on GB300.

One JSON line (rank 0).  Headline `value`: chunkwise-prefill tokens/s on the
32K-token, 96-head, d=128 bf16 workload, inputs resident in HBM, one
kda_chunk_fwd call per step (its two-kernel form: chunk slot list, chunk-local
kernel, state walk).  Extra keys measured in the same run:
  "verify": fused verify-replay on 256 requests x 96 heads (state GB/s, % HBM)
  "verify_ragged": the same with 3..7 drafts per request (ragged entry point)
  "verify_latency": one call at 1 request x 12 heads, 4 positions, from a
            CUDA graph of 20 calls
  "backward": the backward of the headline prefill (dq, dk, dv, dg, dbeta)
            and its training pair (forward keeping its operands, reverse pass)
  "ckpt":   the headline prefill also emitting the state every 4096 tokens
  "decode": the same entry point as single-token decode (window 0) on 256 x 96
  "varlen": 16 packed sequences (1K-8K tokens) continuing from stored states
  "cp":     1M-token, 12-head prefill with the context-parallel schedule,
            its backward over the same segments and that training pair
  "roofline" (the step's dominant kernel), "path_roofline", "kernels",
  "cpu_baseline", "e2e" (host buffers through kda_chunk_fwd_host), "clocks",
  "gpu_launches".

--impl reference times the fp64 CPU oracle (the reference arm of this
repository) on a bounded sample of the same workload.

Multi-GPU (torchrun): independent replicas, one per rank (the recurrence needs
no exchange step when heads and sequences are the work units); time = max over
ranks, value = all ranks' tokens / that time.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA prefill tok/s @H96 d128 (% TC peak); spec-verify state GB/s (% HBM)"
BYTES_PER_TOKHEAD = 1540        # q,k,v bf16 768 + g fp32 512 + beta 4 + o bf16 256 (dk=dv=128)
FLOPS_PER_TOKHEAD_ALGO = 139264  # 3*C*dk + 2*C*dv + 6*dk*dv, C=64, causal halves only
BLOB_PER_TOKHEAD = 66048 / 64    # operand blob of a (chunk, head) handed from the chunk-local kernel to the walk
# bytes per token-head each prefill kernel must move: what it reads and writes at the minimum
KERNEL_BYTES_PER_TOKHEAD = {
    "kda_chunk_prep_kernel": 2 * 128 * 2 + 128 * 4 + 4 + BLOB_PER_TOKHEAD,  # q, k, g, beta in; blob out
    "kda_chunk_walk_kernel": BLOB_PER_TOKHEAD + 128 * 2 + 128 * 2,           # blob, v in; o out
    "kda_chunk_tc_kernel": BYTES_PER_TOKHEAD,
    "kda_chunk_kernel": BYTES_PER_TOKHEAD,
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_traffic(kernel_key, T):
    """DRAM bytes per launch of `kernel_key` from the committed ncu summary,
    scaled to T tokens (requests, for the verify kernel), or None when the
    kernel source changed since."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel_key]
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != rec["source_sha256_16"]:
                return None
        return rec["traffic_bytes_captured"] * T / rec.get("captured_T", rec.get("captured_R"))
    except Exception:
        return None


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x, ws):
    """Max over ranks (identity at world size 1)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        sm.sort()
        med = sm[len(sm) // 2] if sm else None
        return {"sm_mhz": med, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


def cuda_time(fn, steps, stream):
    """Mean ms per call, CUDA events on `stream`, synchronised on both sides."""
    import torch
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(steps):
        fn()
    e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / steps


def timed_launches(kda, fn, steps, stream):
    """cuda_time of `steps` calls with the library's launch timing on: returns
    (mean ms per call, {kernel family: {"launches", "ms"}} over those calls)."""
    kda.kernel_timing_start()
    try:
        ms = cuda_time(fn, steps, stream)
    finally:
        kern = kda.kernel_timing_stop()
    return ms, kern


def cpu_baseline_sample(nthreads=0):
    """The oracle as it stands on a bounded sample of the prefill workload:
    all 96 heads of the first 4096 tokens of the 32K sequence."""
    import numpy as np
    import torch

    import oracle
    from kda_gated_delta_02_gb300 import synth
    oracle.build()
    Ts = 4096
    w = synth.PREFILL_32K
    inp = synth.make_prefill(w, device="cpu", T_override=Ts)
    to = lambda t: t.double().numpy()
    args = [to(inp[k]) for k in ("q", "k", "v", "g", "beta")]
    cu = np.array([0, Ts], dtype=np.int32)
    t0 = time.perf_counter()
    oracle.prefill(*args, cu, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return {"value": Ts / dt, "unit": "tok/s", "cores": oracle.max_threads() if nthreads <= 0 else nthreads,
            "kind": "oracle", "seconds": dt,
            "sample": f"first {Ts} tokens x all {w.H} heads of the T=32768 H=96 d=128 prefill (fp64, OpenMP over heads)",
            "cpu": platform.processor() or platform.machine(), "nproc": os.cpu_count()}


def prefill_config(ws):
    """The `config` of the headline line (both arms)."""
    from kda_gated_delta_02_gb300 import synth
    w = synth.PREFILL_32K
    return {"workload": w.name, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv, "chunk": 64, "global_batch": 1,
            "seq_len": w.T, "parallelism": f"replicas x{ws}",
            "l2": "inputs (4.8 GB) larger than L2 (129 MB); no flush"}


def run_reference(args):
    ws, rank, _ = dist_info()
    if rank != 0:
        return 0
    steps = max(1, args.steps)
    res = None
    total_t, total_tok = 0.0, 0
    for _ in range(max(0, args.warmup)):
        pass  # the oracle has no warm-up state; warm-up steps are skipped
    for _ in range(steps):
        res = cpu_baseline_sample()
        total_t += res["seconds"]
        total_tok += res["value"] * res["seconds"]
    value = total_tok / total_t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": dict(prefill_config(ws), sample_tokens=4096,
                           sample="first 4096 tokens of the workload, all heads, per step"),
            "cpu_baseline": {"kind": "oracle", "cores": res["cores"], "sample": res["sample"], "value": value,
                             "unit": "tok/s"},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def verify_kernel_name():
    return "kda_verify_tc_kernel"


def decode_workload(synth):
    """Single-token decode: 256 requests x 96 heads, d = 128, conv width 4, no draft window."""
    return synth.DecodeWorkload("decode R=256 H=96 d=128 W=4 one token (window 0)", 256, 96, 128, 128,
                                Wd=0, seed=5)


def run_profile(args):
    """Plain launches of one kernel family on a chosen size (for ncu captures)."""
    import torch
    torch.cuda.set_device(0)
    from kda_gated_delta_02_gb300 import build as kbuild
    kbuild.build()
    import kda_gated_delta_02_gb300 as kda
    from kda_gated_delta_02_gb300 import synth
    n = max(1, args.warmup) + max(1, args.steps)
    if args.profile == "backward":
        inp = synth.make_prefill(synth.PREFILL_32K, device="cuda", T_override=args.T or None)
        dout = torch.randn(inp["v"].shape, dtype=torch.float32, device="cuda").to(inp["v"].dtype)
        for _ in range(n):
            kda.chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["cu_seqlens"], dout)
        torch.cuda.synchronize()
        print(f"profile {args.profile}: {n} launches ok")
        return 0
    if args.profile in ("prefill", "cp"):
        w = synth.PREFILL_32K if args.profile == "prefill" else synth.ULTRA_LONG
        inp = synth.make_prefill(w, device="cuda", T_override=args.T or None)
        for _ in range(n):
            kda.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["cu_seqlens"],
                          cp_mode=kda.CP_AUTO if args.profile == "cp" else kda.CP_OFF)
    else:
        dw = synth.VERIFY if args.profile == "verify" else decode_workload(synth)
        R = args.R or dw.R
        d = synth.make_decode(dw, device="cuda", R_override=R,
                              accepted=None if args.profile == "verify" else [0] * R)
        for _ in range(n):
            kda.decode_verify_replay(d["state"], d["tail"], d["conv_w"], d["cached_qkv"], d["cached_g"],
                                     d["cached_b"], d["accepted"], d["new_qkv"], d["new_g"], d["new_b"],
                                     d["out_w"])
    torch.cuda.synchronize()
    print(f"profile {args.profile}: {n} launches ok")
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kda", choices=["kda", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default="", help="comma list of prefill,verify,decode,varlen,cp,backward (default: all)")
    ap.add_argument("--profile", default="", choices=["", "prefill", "verify", "decode", "cp", "backward"],
                    help="launch only this kernel family (warmup + steps launches, no JSON) for ncu")
    ap.add_argument("--T", type=int, default=0, help="token count override for --profile prefill/cp/backward")
    ap.add_argument("--R", type=int, default=0, help="request count override for --profile verify/decode")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile(args)

    import torch
    ws, rank, local = dist_info()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    from kda_gated_delta_02_gb300 import build as kbuild
    kbuild.build()
    import kda_gated_delta_02_gb300 as kda
    from kda_gated_delta_02_gb300 import synth
    kda.load_library()
    peaks = load_peaks()
    only = set(args.only.split(",")) if args.only else {"prefill", "verify", "decode", "varlen", "cp", "backward"}
    K, Wm = max(1, args.steps), max(3, args.warmup)
    stream = torch.cuda.current_stream()
    out = {}

    # ------------------------------------------------------------ prefill (headline)
    # dk = dv = 128 bf16 with the workspace of the two-kernel form: per step the
    # chunk-local kernel and the walk, once per piece of slots
    w = synth.PREFILL_32K
    inp = synth.make_prefill(w, device="cuda")
    T, H = inp["q"].shape[:2]
    o = torch.empty_like(inp["v"])
    Sf = torch.empty((1, H, w.dk, w.dv), dtype=torch.float32, device="cuda")
    wsp = torch.empty(max(1, kda.chunk_fwd_prep_workspace_size(1, T, H, w.dk, w.dv, kda.CP_AUTO)),
                      dtype=torch.uint8, device="cuda")

    def prefill_step():
        kda.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["cu_seqlens"], out=o,
                      final_state=Sf, cp_mode=kda.CP_AUTO, workspace=wsp)

    for _ in range(Wm):
        prefill_step()
    sampler = ClockSampler(local)
    sampler.start()
    barrier(ws)
    ms = cuda_time(prefill_step, K, stream)
    barrier(ws)
    clocks = sampler.stop()
    ms = reduce_max(ms, ws)
    # Per-kernel launch times come from a second timed pass with the library's
    # launch events on: an event between a walk and the chunk-local launch that
    # follows it as a programmatic dependent serialises the two, so these are
    # the kernels' own durations without the overlap of the headline pass.
    ms_ev, kern = timed_launches(kda, prefill_step, K, stream)
    tok_s = ws * T / (ms * 1e-3)
    path_bytes = T * H * BYTES_PER_TOKHEAD + H * w.dk * w.dv * 4
    path_gbs = path_bytes / (ms * 1e-3) / 1e9
    algo_flops = T * H * FLOPS_PER_TOKHEAD_ALGO
    tflops = algo_flops / (ms * 1e-3) / 1e12
    per_step_launches = sum(v["launches"] for v in kern.values()) / K
    launches = int(round(2 * K * per_step_launches))  # the headline pass and the launch-events pass
    # the dominant kernel of the step: its average launch (events on the launching
    # stream, inside the timed region) against the bytes it must move per launch
    kernels = {}
    for name, v in kern.items():
        per_step = v["launches"] / K
        lms = v["ms"] / v["launches"]
        rec = {"launches_per_step": per_step, "ms_per_launch": lms, "share_of_step": v["ms"] / K / ms_ev}
        if name in KERNEL_BYTES_PER_TOKHEAD:
            tokens = T / per_step  # tokens one launch covers
            rec["bytes_per_launch"] = tokens * H * KERNEL_BYTES_PER_TOKHEAD[name]
            rec["achieved_gbs"] = rec["bytes_per_launch"] / (lms * 1e-3) / 1e9
            rec["frac_hbm"] = rec["achieved_gbs"] / peaks["hbm_gbs"]
            rec["traffic"] = kernel_traffic(name, tokens)
        kernels[name] = rec
    dom = max((n for n in kernels if n in KERNEL_BYTES_PER_TOKHEAD), key=lambda n: kernels[n]["share_of_step"])
    # the roofline of the dominant kernel counts the path's own 1,540 B per
    # token-head for the token-heads one launch covers (what the method must
    # move), not the kernel's own reads and writes of intermediates
    dom_tokens = T / kernels[dom]["launches_per_step"]
    dom_algo = dom_tokens * H * BYTES_PER_TOKHEAD
    dom_gbs = dom_algo / (kernels[dom]["ms_per_launch"] * 1e-3) / 1e9
    # DRAM bytes per step (ncu, committed captures) against the path's bytes
    step_traffic = 0.0
    for name, rec in kernels.items():
        if name in KERNEL_BYTES_PER_TOKHEAD:
            step_traffic = None if (step_traffic is None or rec["traffic"] is None) else \
                step_traffic + rec["traffic"] * rec["launches_per_step"]
    out["prefill"] = {"ms": ms, "tok_s": tok_s}
    out["prefill_launch_events"] = {"ms_per_step": ms_ev,
                                    "note": "launch events on: the chunk-local/walk overlap is serialised"}

    # the same launch emitting the state every 4096 tokens (8 checkpoints per head)
    every = 4096
    ck = torch.empty((1, T // every, H, w.dk, w.dv), dtype=torch.float32, device="cuda")

    def ckpt_step():
        kda.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["cu_seqlens"], out=o,
                      final_state=Sf, cp_mode=kda.CP_AUTO, ckpt_every=every, ckpt=ck)

    for _ in range(2):
        ckpt_step()
    ms_ck = reduce_max(cuda_time(ckpt_step, K, stream), ws)
    out["ckpt"] = {"workload": f"{w.name}, state every {every} tokens", "ms": ms_ck,
                   "tok_s": ws * T / (ms_ck * 1e-3), "overhead_vs_plain": ms_ck / ms - 1.0,
                   "checkpoint_bytes_per_launch": ck.numel() * 4}
    launches += int(round(K * per_step_launches))  # the same launches as the plain step
    del ck

    # e2e: host buffers (page-locked) through the host-buffer C-ABI call, which
    # copies the inputs in and o and the final state out by pieces overlapped
    # with the kernels; every copy is inside the timed region
    host = {k: v.to("cpu").pin_memory() for k, v in inp.items() if v is not None}
    host["cu_seqlens"] = inp["cu_seqlens"].cpu()
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    Sf_host = torch.empty(Sf.shape, dtype=Sf.dtype).pin_memory()
    e2e_pieces = 8
    wsh = torch.empty(kda.load_library().kda_chunk_fwd_host_workspace_size(1, T, H, w.dk, w.dv, 0, e2e_pieces),
                      dtype=torch.uint8, device="cuda")
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = o_host.numel() * o_host.element_size() + Sf_host.numel() * Sf_host.element_size()

    def e2e_step():
        kda.chunk_fwd_host(host["q"], host["k"], host["v"], host["g"], host["beta"], host["cu_seqlens"],
                           out=o_host, final_state=Sf_host, pieces=e2e_pieces, workspace=wsh)

    e2e_step()
    Ke = max(3, K // 4)
    ms_e2e = reduce_max(cuda_time(e2e_step, Ke, stream), ws)
    del host, o_host, Sf_host, wsh
    del inp, o, wsp
    torch.cuda.empty_cache()

    # ------------------------------------------------------------ verify-replay
    if "verify" in only:
        vw = synth.VERIFY
        verify_kernel = verify_kernel_name()
        d = synth.make_decode(vw, device="cuda")
        st, tl = d["state"].clone(), d["tail"].clone()
        ov = torch.empty((vw.R, vw.Wd + 1, vw.H, vw.dv), dtype=torch.bfloat16, device="cuda")

        def verify_step():
            kda.decode_verify_replay(st, tl, d["conv_w"], d["cached_qkv"], d["cached_g"], d["cached_b"],
                                     d["accepted"], d["new_qkv"], d["new_g"], d["new_b"], d["out_w"], out=ov)

        for _ in range(Wm):
            verify_step()
        vms, kv = timed_launches(kda, verify_step, K, stream)
        vms = reduce_max(vms, ws)
        state_bytes = 2 * st.numel() * st.element_size()  # read + write
        acc = d["accepted"].to(torch.int64)
        row = 3 * vw.H * vw.dk * 2 + vw.H * vw.dk * 2 + vw.H * 2  # pre-conv qkv + g + beta per token row
        proj_bytes = int((acc.sum().item() + vw.R * (vw.Wd + 1)) * row)
        tail_bytes = 2 * tl.numel() * tl.element_size()
        o_bytes = ov.numel() * ov.element_size()
        total_bytes = state_bytes + proj_bytes + tail_bytes + o_bytes
        out["verify"] = {"workload": vw.name, "ms": vms, "state_gbs": ws * state_bytes / (vms * 1e-3) / 1e9,
                         "total_gbs": ws * total_bytes / (vms * 1e-3) / 1e9,
                         "frac_hbm": (total_bytes / (vms * 1e-3) / 1e9) / peaks["hbm_gbs"],
                         "bytes_per_launch": total_bytes, "state_bytes_per_launch": state_bytes,
                         "kernel": verify_kernel, "traffic": kernel_traffic(verify_kernel, vw.R),
                         "requests_per_s": ws * vw.R / (vms * 1e-3)}
        launches += sum(v["launches"] for v in kv.values())
        del d, st, tl, ov
        torch.cuda.empty_cache()

    # ------------------------------------------------------------ backward (training), same workload
    if "backward" in only:
        inp = synth.make_prefill(w, device="cuda")
        dout = torch.randn(inp["v"].shape, dtype=torch.float32, device="cuda").to(inp["v"].dtype)
        bws = torch.empty(kda.load_library().kda_chunk_bwd_workspace_size(1, T, H, w.dk, w.dv), dtype=torch.uint8,
                          device="cuda")

        def bwd_step():
            kda.chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["cu_seqlens"], dout,
                          workspace=bws)

        bwd_step()
        tc_form = w.dk == 128 and inp["q"].dtype == torch.bfloat16
        Kb = max(3, K // 4) if tc_form else max(2, K // 10)
        bms = reduce_max(cuda_time(bwd_step, Kb, stream), ws)
        _, kb = timed_launches(kda, bwd_step, Kb, stream)  # kernel table (launch events add gaps)
        kb_total = sum(v["ms"] for v in kb.values())
        bkern = {name: {"launches_per_step": v["launches"] / Kb, "ms_per_launch": v["ms"] / max(v["launches"], 1),
                        "share_of_step": v["ms"] / max(kb_total, 1e-9)} for name, v in kb.items()}
        # algorithmic I/O per token-head: q, k, v, do bf16 + g, beta in; dq, dk, dv, dg, dbeta fp32 out
        io = T * H * (4 * 128 * 2 + 128 * 4 + 4 + 3 * 128 * 4 + 128 * 4 + 4)
        entry = {"workload": w.name + " backward (dq, dk, dv, dg, dbeta)", "ms": bms,
                 "tok_s": ws * T / (bms * 1e-3), "algorithmic_bytes_per_step": io,
                 "frac_hbm": io / (bms * 1e-3) / 1e9 / peaks["hbm_gbs"], "ratio_to_forward": bms / ms,
                 "kernels": bkern}
        if tc_form:
            # tensor-core products issued per (chunk, head), padding included:
            # forward pass (A/B tiles 128x160x128, W 128x64x64, walk U 128x64x(64+128),
            # state 128x128x64), reverse walk (dU 128x64x(64+128), dS 2 x 128x128x64)
            # and the chunk kernel (batches of 128x64x128, 2 x 128x64x64, 2 x 128x128x128,
            # 128x64x128, 2 x 128x64x64, 2 x (128x128x160 + 128x160x128))
            macs = (128 * 160 * 128 + 128 * 64 * 64 + 128 * 64 * 192 + 128 * 128 * 64 +
                    128 * 64 * 192 + 2 * 128 * 128 * 64 +
                    128 * 64 * 128 + 2 * 128 * 64 * 64 + 2 * 128 * 128 * 128 + 128 * 64 * 128 +
                    2 * 128 * 64 * 64 + 2 * (128 * 128 * 160 + 128 * 160 * 128))
            flops = 2.0 * macs * (T // 64) * H
            entry.update({"form": "chunk (WY) form on the tensor cores",
                          "tensor_tflops_issued": flops / (bms * 1e-3) / 1e12,
                          "tensor_frac": flops / (bms * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"],
                          "workspace_bytes": int(bws.numel())})
            # the training pair: the forward keeps its operands, the backward
            # is the reverse pass alone (a training step runs each once)
            def fwd_train():
                kda.chunk_fwd_train(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["cu_seqlens"],
                                    saved=bws)

            def bwd_saved():
                kda.chunk_bwd_saved(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["cu_seqlens"], dout,
                                    bws)

            fwd_train()
            bwd_saved()
            fms = reduce_max(cuda_time(fwd_train, Kb, stream), ws)
            sms = reduce_max(cuda_time(bwd_saved, Kb, stream), ws)
            entry["training_pair"] = {
                "fwd_train_ms": fms, "fwd_train_vs_forward": fms / ms,
                "bwd_saved_ms": sms, "bwd_saved_vs_forward": sms / ms,
                "step_ms": fms + sms,
                "note": "kda_chunk_fwd_train (prefill outputs + the operands the backward needs) then "
                        "kda_chunk_bwd_saved (reverse pass only); same results as kda_chunk_fwd / kda_chunk_bwd"}
        else:
            entry["form"] = "token-level reverse mode on the CUDA cores"
        out["backward"] = entry
        launches += sum(v["launches"] for v in kb.values())
        del inp, dout, bws
        torch.cuda.empty_cache()

    # ------------------------------------------------------------ ragged verify (drafts 3..7 per request)
    if "verify" in only:
        import numpy as np
        rg = np.random.default_rng(3)
        rw = synth.DecodeWorkload("verify-replay ragged R=256 H=96 d=128 W=4, window 7, drafts U{3..7}",
                                  256, 96, 128, 128, Wd=7, seed=4)
        d = synth.make_decode(rw, device="cuda")
        dl = torch.as_tensor(rg.integers(3, 8, size=rw.R), dtype=torch.int32, device="cuda")
        st, tl = d["state"].clone(), d["tail"].clone()
        ov = torch.empty((rw.R, rw.Wd + 1, rw.H, rw.dv), dtype=torch.bfloat16, device="cuda")

        def ragged_step():
            kda.decode_verify_replay(st, tl, d["conv_w"], d["cached_qkv"], d["cached_g"], d["cached_b"],
                                     d["accepted"], d["new_qkv"], d["new_g"], d["new_b"], d["out_w"], out=ov,
                                     draft_len=dl)

        for _ in range(Wm):
            ragged_step()
        rms, kr = timed_launches(kda, ragged_step, K, stream)
        rms = reduce_max(rms, ws)
        tokens = int((d["accepted"].to(torch.int64) + 1 + dl.to(torch.int64)).sum().item())
        out["verify_ragged"] = {"workload": rw.name, "ms": rms, "requests_per_s": ws * rw.R / (rms * 1e-3),
                                "tokens_replayed_per_launch": tokens,
                                "state_gbs": ws * 2 * st.numel() * st.element_size() / (rms * 1e-3) / 1e9}
        launches += sum(v["launches"] for v in kr.values())
        del d, st, tl, ov, dl
        torch.cuda.empty_cache()

        # latency of one small call, the shape the pages measure their verify
        # kernel on (one sequence, 96 / 8 = 12 heads per tensor-parallel rank,
        # 4 verify positions), replayed from a CUDA graph of 20 calls
        sw = synth.DecodeWorkload("verify-replay latency R=1 H=12 d=128 W=4, 4 positions (bonus + 3 drafts)",
                                  1, 12, 128, 128, Wd=3, seed=6)
        d = synth.make_decode(sw, device="cuda")
        st, tl = d["state"].clone(), d["tail"].clone()
        ov = torch.empty((sw.R, sw.Wd + 1, sw.H, sw.dv), dtype=torch.bfloat16, device="cuda")

        def small_step():
            kda.decode_verify_replay(st, tl, d["conv_w"], d["cached_qkv"], d["cached_g"], d["cached_b"],
                                     d["accepted"], d["new_qkv"], d["new_g"], d["new_b"], d["out_w"], out=ov)

        gs = torch.cuda.Stream()
        gs.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(gs):
            small_step()
            gs.synchronize()
            with torch.cuda.graph(graph, stream=gs):
                for _ in range(20):
                    small_step()
        torch.cuda.synchronize()
        for _ in range(Wm):
            graph.replay()
        lus = reduce_max(cuda_time(graph.replay, K, stream), ws) * 1e3 / 20
        out["verify_latency"] = {"workload": sw.name, "us_per_call": lus, "calls_per_graph": 20,
                                 "pages_number": {"us_per_layer": 5.61, "hardware": "AMD MI355X",
                                                  "note": "the pages' optimised verify kernel, other hardware: "
                                                          "context, not a target"}}
        launches += 20 * K
        del d, st, tl, ov, graph
        torch.cuda.empty_cache()

    # ------------------------------------------------------------ single-token decode (window 0)
    if "decode" in only:
        dw = decode_workload(synth)
        decode_kernel = "kda_decode_token_kernel<128>"
        d = synth.make_decode(dw, device="cuda", accepted=[0] * dw.R)
        st, tl = d["state"].clone(), d["tail"].clone()
        od = torch.empty((dw.R, 1, dw.H, dw.dv), dtype=torch.bfloat16, device="cuda")

        def decode_step():
            kda.decode_verify_replay(st, tl, d["conv_w"], d["cached_qkv"], d["cached_g"], d["cached_b"],
                                     d["accepted"], d["new_qkv"], d["new_g"], d["new_b"], d["out_w"], out=od)

        for _ in range(Wm):
            decode_step()
        dms, kd = timed_launches(kda, decode_step, K, stream)
        dms = reduce_max(dms, ws)
        state_bytes = 2 * st.numel() * st.element_size()
        row = 3 * dw.H * dw.dk * 2 + dw.H * dw.dk * 2 + dw.H * 2
        total_bytes = state_bytes + dw.R * row + 2 * tl.numel() * tl.element_size() + od.numel() * od.element_size()
        out["decode"] = {"workload": dw.name, "ms": dms, "state_gbs": ws * state_bytes / (dms * 1e-3) / 1e9,
                         "frac_hbm": (total_bytes / (dms * 1e-3) / 1e9) / peaks["hbm_gbs"],
                         "bytes_per_launch": total_bytes, "tokens_per_s": ws * dw.R / (dms * 1e-3),
                         "kernel": decode_kernel, "traffic": kernel_traffic(decode_kernel, dw.R)}
        launches += sum(v["launches"] for v in kd.values())
        del d, st, tl, od
        torch.cuda.empty_cache()

    # ------------------------------------------------------------ varlen prefix continuation
    if "varlen" in only:
        vl = synth.VARLEN
        vi = synth.make_prefill(vl, device="cuda")
        Tv, Hv = vi["q"].shape[:2]
        ov = torch.empty_like(vi["v"])
        Sv = torch.empty_like(vi["S0"])

        def varlen_step():
            kda.chunk_fwd(vi["q"], vi["k"], vi["v"], vi["g"], vi["beta"], vi["cu_seqlens"],
                          initial_state=vi["S0"], out=ov, final_state=Sv, cp_mode=kda.CP_AUTO)

        for _ in range(3):
            varlen_step()
        Kv = max(3, K // 2)
        vms_, kl = timed_launches(kda, varlen_step, Kv, stream)
        vms_ = reduce_max(vms_, ws)
        vbytes = Tv * Hv * BYTES_PER_TOKHEAD + 2 * vi["S0"].numel() * 4
        out["varlen"] = {"workload": vl.name, "tokens": Tv, "ms": vms_, "tok_s": ws * Tv / (vms_ * 1e-3),
                         "frac_hbm": (vbytes / (vms_ * 1e-3) / 1e9) / peaks["hbm_gbs"]}
        launches += sum(v["launches"] for v in kl.values())
        del vi, ov, Sv
        torch.cuda.empty_cache()

    # ------------------------------------------------------------ ultra-long, context parallel
    if "cp" in only:
        cw = synth.ULTRA_LONG
        ci = synth.make_prefill(cw, device="cuda")
        Tc, Hc = ci["q"].shape[:2]
        oc = torch.empty_like(ci["v"])
        Sc = torch.empty((1, Hc, cw.dk, cw.dv), dtype=torch.float32, device="cuda")
        seg = kda.chunk_fwd_plan(1, Tc, Hc, cw.dk, cw.dv, kda.CP_AUTO)
        wsb = kda.chunk_fwd_prep_workspace_size(1, Tc, Hc, cw.dk, cw.dv, kda.CP_AUTO)
        wbuf = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")

        def cp_step(mode=kda.CP_AUTO):
            kda.chunk_fwd(ci["q"], ci["k"], ci["v"], ci["g"], ci["beta"], ci["cu_seqlens"], out=oc,
                          final_state=Sc, cp_mode=mode, workspace=wbuf)

        for _ in range(3):
            cp_step()
        Kc = max(3, K // 4)
        cms, kcp = timed_launches(kda, cp_step, Kc, stream)
        cms = reduce_max(cms, ws)
        cms_off = reduce_max(cuda_time(lambda: cp_step(kda.CP_OFF), 1, stream), ws)
        minimal = Tc * Hc * BYTES_PER_TOKHEAD
        # the CP schedule's own bytes: the minimum plus its transition pass's
        # second read of k, v, g and beta (768 - 256 + 512 + 4 B per token-head)
        cp_bytes = Tc * Hc * (BYTES_PER_TOKHEAD + 1028)
        out["cp"] = {"workload": cw.name, "segment_len": seg, "ms": cms, "tok_s": ws * Tc / (cms * 1e-3),
                     "ms_cp_off": cms_off, "speedup_vs_off": cms_off / cms,
                     "frac_hbm_min_bytes": (minimal / (cms * 1e-3) / 1e9) / peaks["hbm_gbs"],
                     "frac_hbm_cp_bytes": (cp_bytes / (cms * 1e-3) / 1e9) / peaks["hbm_gbs"],
                     "cp_bytes_per_tokhead": BYTES_PER_TOKHEAD + 1028}
        launches += sum(v["launches"] for v in kcp.values())
        del oc, wbuf
        torch.cuda.empty_cache()
        if "backward" in only and cw.dk == 128 and ci["q"].dtype == torch.bfloat16:
            # the backward of the same call over context-parallel segments
            dco = torch.randn(ci["v"].shape, dtype=torch.float32, device="cuda").to(ci["v"].dtype)
            lib = kda.load_library()
            bneed = lib.kda_chunk_bwd_cp_workspace_size(1, Tc, Hc, cw.dk, cw.dv, kda.CP_AUTO, 0)
            bwb = torch.empty(max(bneed, 1), dtype=torch.uint8, device="cuda")

            def cpb_step(mode=kda.CP_AUTO):
                kda.chunk_bwd_cp(ci["q"], ci["k"], ci["v"], ci["g"], ci["beta"], ci["cu_seqlens"], dco,
                                 cp_mode=mode, workspace=bwb, want_dS0=False)

            cpb_step()
            Kcb = max(3, K // 8)
            cbms = reduce_max(cuda_time(cpb_step, Kcb, stream), ws)
            _, kcb = timed_launches(kda, cpb_step, Kcb, stream)  # kernel table (launch events add gaps)
            cbms_off = reduce_max(cuda_time(lambda: cpb_step(kda.CP_OFF), 1, stream), ws)
            kcb_total = sum(v["ms"] for v in kcb.values())
            out["cp"]["backward"] = {
                "ms": cbms, "tok_s": ws * Tc / (cbms * 1e-3), "ratio_to_forward": cbms / cms,
                "ms_cp_off": cbms_off, "speedup_vs_off": cbms_off / cbms, "workspace_bytes": int(bwb.numel()),
                "segments": "automatic: about one (segment, head) unit per SM for the reverse walks",
                "kernels": {name: {"launches_per_step": v["launches"] / Kcb,
                                   "share_of_step": v["ms"] / max(kcb_total, 1e-9)} for name, v in kcb.items()}}
            launches += sum(v["launches"] for v in kcb.values())

            def cp_fwd_train():
                kda.chunk_fwd_train(ci["q"], ci["k"], ci["v"], ci["g"], ci["beta"], ci["cu_seqlens"], saved=bwb,
                                    cp_mode=kda.CP_AUTO)

            def cp_bwd_saved():
                kda.chunk_bwd_saved(ci["q"], ci["k"], ci["v"], ci["g"], ci["beta"], ci["cu_seqlens"], dco, bwb,
                                    cp_mode=kda.CP_AUTO, want_dS0=False)

            cp_fwd_train()
            cp_bwd_saved()
            tfms = reduce_max(cuda_time(cp_fwd_train, Kcb, stream), ws)
            tbms = reduce_max(cuda_time(cp_bwd_saved, Kcb, stream), ws)
            out["cp"]["backward"]["training_pair"] = {
                "fwd_train_ms": tfms, "fwd_train_vs_forward": tfms / cms,
                "bwd_saved_ms": tbms, "bwd_saved_vs_forward": tbms / cms, "step_ms": tfms + tbms,
                "note": "kda_chunk_fwd_train_cp then kda_chunk_bwd_saved_cp (reverse pass only); same results as "
                        "kda_chunk_fwd / kda_chunk_bwd_cp"}
            del dco, bwb
        del ci
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_sample()
        cpu.pop("seconds", None)

    if rank == 0:
        line = {
            "metric": METRIC, "value": tok_s, "unit": "tok/s", "n_gpus": ws, "steps": K, "warmup": Wm,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded torch generator, shapes of the pages' workloads)",
            "config": prefill_config(ws),
            "roofline": {"bound": "hbm", "achieved": dom_gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": dom_gbs / peaks["hbm_gbs"], "traffic": kernels[dom]["traffic"],
                         "peak_source": peaks["source"], "kernel": dom,
                         "algorithmic_bytes_per_launch": dom_algo,
                         "algorithmic_bytes_per_tokhead": BYTES_PER_TOKHEAD,
                         "tokheads_per_launch": dom_tokens * H,
                         "ms_per_launch": kernels[dom]["ms_per_launch"],
                         "kernel_own_bytes_per_launch": kernels[dom]["bytes_per_launch"],
                         "kernel_own_frac": kernels[dom]["frac_hbm"]},
            "path_roofline": {"bound": "hbm", "achieved": path_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "frac": path_gbs / peaks["hbm_gbs"], "algorithmic_bytes_per_step": path_bytes,
                              "dram_traffic_per_step": step_traffic,
                              "traffic_ratio": None if step_traffic is None else step_traffic / path_bytes,
                              "tensor_tflops": tflops, "tensor_peak_tflops": peaks["bf16_tflops"],
                              "tensor_frac": tflops / peaks["bf16_tflops"]},
            "kernels": kernels,
            "e2e": {"value": ws * T / (ms_e2e * 1e-3), "unit": "tok/s", "ms": ms_e2e,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "call": f"kda_chunk_fwd_host, {e2e_pieces} pieces"},
            "clocks": clocks, "gpu_launches": launches,
        }
        line.update({k: v for k, v in out.items() if k != "prefill"})
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
