"""Benchmark of the CSA2 decode hot path on GB300.

One step = one Full-layer decode of a batch: lightning-indexer scores over
every cache entry -> top-512 -> sparse MQA attention over the 512 selected FP4
entries plus the 128-entry FP8 window.  Default workload: 8 sequences x
1,048,576-entry m=1 caches with Zipf-skewed indexer keys, one query token per
sequence (the 1M-context decode the metric is quoted on).

Prints ONE JSON line (rank 0).  Timing: W untimed warm-up steps, then K steps
between CUDA events on the launching stream, barrier + synchronize on both
sides, max over ranks.  Each step streams 573 MB of cache (far more than the
129 MB L2), so no extra L2 flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config 4] [--no-cpu-baseline]

--config 0/1/4 time other Full-layer decode batches the same way.  --config 3
(Reindex decode: 64 x 1,048,576 entries, pool of 2,048 blocks given) and
--config 2 (m=2 chunked prefill: 8,192 causal queries over 4,096 pooled
entries) time those steps and report the roofline of their dominant kernel
(the pool-mode indexer against HBM; the attention against the bf16 tensor
peak); they are measurements of those steps, not the headline line.

--impl reference times the CPU oracle (plain C, fp64) on the host cores on a
bounded sample of the same workload; under torchrun only rank 0 runs it.
Multi-GPU (torchrun): every rank decodes its own batch on its own GPU (the
batches are independent, no data-path collective): weak scaling.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode query-tokens/s for CSA2 (score+top512+attn) at 1M ctx; HBM GB/s vs peak"
UNIT = "query-tokens/s"
FIXED_BYTES_PER_QUERY = 348_416      # 512x288 + 128x528 + q 64 KiB + out 64 KiB + q_idx 2176 + w 128
IDX_BYTES = 68


# dram__bytes_read.sum + dram__bytes_write.sum of one index_score_tc_kernel launch inside
# csa2_decode, from an ncu capture (--metrics dram__bytes_read.sum,dram__bytes_write.sum) of the
# current kernel on the named workload; workloads without such a capture report null.
INDEX_SCORE_TRAFFIC = {"long_full_decode_N1M_B8_zipf": 570_488_832 + 4_995_328,
                       "full_decode_N65536_B32": 142_722_048 + 4_186_880,
                       "reindex_decode_N1M_B64": 84_265_984 + 1_812_480}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="with the default workload, skip the secondary workloads")
    ap.add_argument("--entries", type=int, default=None,
                    help="shorten the workload's caches to this many entries per sequence (smaller device "
                         "footprint, e.g. for profiler captures); the workload name records it")
    ap.add_argument("--only", choices=["mq", "layers", "build"], default=None,
                    help="run and print only one secondary workload: the multi-query decode (mq), the "
                         "20-layer decoder step (layers) or the cache build of a 1M-token prompt (build)")
    return ap.parse_args()


def workload_of(args):
    """The configuration's workload, its caches shortened to --entries if given."""
    import dataclasses
    from gen.workloads import CONFIGS
    wl = CONFIGS[args.config]
    if args.entries is not None and args.entries != wl.n_entries:
        wl = dataclasses.replace(wl, n_entries=args.entries, name=f"{wl.name}_entries{args.entries}")
    return wl


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ------------------------------------------------------------------ CPU oracle
def oracle_decode_sample(wl, qi=0):
    """Time the oracle's decode of one query (score all entries, top-512,
    attention) with its packed caches prepared beforehand (they are resident
    state, not step work)."""
    import numpy as np
    import oracle
    from oracle.compose import packed_keys, kv_records, swa_records, query_inputs
    seq, n = int(wl.q_seq()[qi]), int(wl.n_vis()[qi])
    keys = packed_keys(wl, seq, n)
    qidx, w = query_inputs(wl, qi)
    q = wl.q(qi)
    t0 = time.perf_counter()
    s = oracle.index_score(keys, qidx, w)
    sel = oracle.topk(s, 512)
    t1 = time.perf_counter()
    kv = kv_records(wl, seq, sel[sel >= 0])            # record fetch = the gather of the selected entries
    sw = swa_records(wl, seq, int(wl.swa_first()[qi]), int(wl.swa_cnt()[qi]))
    t2 = time.perf_counter()
    oracle.sparse_attn(q, kv, sw, int(wl.pos()[qi]))
    t3 = time.perf_counter()
    # record generation (t1..t2) is input synthesis, not oracle work
    return (t1 - t0) + (t3 - t2)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(wl, n_samples=1):
    secs = [oracle_decode_sample(wl, qi) for qi in range(n_samples)]
    per_q = sum(secs) / len(secs)
    threads = int(os.environ.get("OMP_NUM_THREADS", cpu_cores()))
    return {"value": 1.0 / per_q, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n_samples} of {wl.n_q} queries (sequence 0), full {wl.n_entries}-entry cache: "
                      f"fp64 score of every entry + top-512 sort + attention, {per_q:.2f} s per query"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    def __init__(self, gpu_index: int):
        import tempfile
        self.path = os.path.join(tempfile.gettempdir(), f"csa2_clocks_{os.getpid()}.csv")
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def staged_inputs(tensors):
    """One pinned host buffer holding the given host tensors (each at a 256-B
    aligned offset), its device twin, and device views of the same shapes and
    dtypes: a step's inputs then travel in one host-to-device copy."""
    import torch
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.zeros(total, dtype=torch.uint8).pin_memory()
    dev = torch.empty(total, dtype=torch.uint8, device="cuda")
    views = []
    for t, o in zip(tensors, offs):
        n = t.numel() * t.element_size()
        host[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
        views.append(dev[o:o + n].view(t.dtype).view(t.shape))
    dev.copy_(host)
    return host, dev, views


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import compressed_sparse_attention_index_gb300 as C
    from compressed_sparse_attention_index_gb300 import decode
    from gen.device import build_device_workload
    from gen.workloads import CONFIGS

    from compressed_sparse_attention_index_gb300 import ranks
    torch.cuda.set_device(local_rank)
    wl = ranks.rank_workload(workload_of(args), rank)       # each rank decodes its own batch
    if wl.pool or wl.prefill:
        return run_rows(args, rank, world, local_rank, wl)
    dw = build_device_workload(wl)
    n_q, n_max = dw.q.shape[0], dw.n_max
    buf = decode.DecodeBuffers(n_q, n_max, out_dtype=C.CSA2_OUT_BF16)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()

    def step():
        decode.fused_decode(dw, buf, None, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert C.csa2_get_device_status() == 0

    # device-timed region: K steps of the one-call decode (csa2_decode)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_index = local_rank
    if os.environ.get("CUDA_VISIBLE_DEVICES"):
        try:
            gpu_index = int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local_rank])
        except ValueError:
            pass
    clocks = ClockSampler(gpu_index)
    time.sleep(0.3)
    ranks.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    ranks.barrier()
    clk = clocks.stop()
    ms = t_start.elapsed_time(t_end)
    assert C.csa2_get_device_status() == 0

    # roofline of the dominant kernel: K further csa2_decode steps with the
    # library's profile events recorded around the indexer launch it makes (the
    # same kernel as in the timed steps, epilogue maxima included)
    score_ms = profiled_indexer_ms(args.steps, stream, lambda: decode.fused_decode(dw, buf, None, stream))
    assert C.csa2_get_device_status() == 0
    ms = ranks.max_over_ranks(ms, device="cuda")

    # end to end through the public API: csa2_decode_host takes the step's
    # inputs (attention query, indexer query in bf16, head weights, per-query
    # descriptors) in pinned host memory, copies each in, packs the indexer
    # query, decodes and copies the bf16 output back, all on the stream
    from gen import inputs as G
    import numpy as np
    qidx_bits = np.concatenate([G.normal_block_bf16(wl.seed, G.S_QIDX, qi, 0, 32, 128) for qi in range(n_q)])
    h_q = dw.q.cpu().pin_memory()
    h_qidx = torch.from_numpy(qidx_bits.view(np.int16)).pin_memory()
    h_w = dw.w.cpu().pin_memory()
    h_desc = torch.stack([dw.q_seq, dw.n_vis, dw.pos, dw.swa_first, dw.swa_cnt]).cpu().contiguous().pin_memory()
    h_out = torch.empty(buf.out.shape, dtype=buf.out.dtype).pin_memory()
    ws_h_bytes = C.csa2_workspace_size(C.CSA2_OP_DECODE_HOST, n_q, n_max, 512)
    ws_h = torch.empty(ws_h_bytes, dtype=torch.uint8, device="cuda")
    n_seq = dw.kv.shape[0]

    def e2e_step():
        C.csa2_decode_host(dw.key_nib, dw.key_scale, n_max, n_seq, dw.kv, dw.swa, dw.swa.shape[1], h_q, h_qidx, h_w,
                           h_desc, n_q, None, h_out, C.CSA2_OUT_BF16, None, ws_h, ws_h_bytes, stream)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    assert C.csa2_get_device_status() == 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = ranks.max_over_ranks(e2e_ms, device="cuda")
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_qidx, h_w, h_desc))
    d2h = h_out.numel() * h_out.element_size()
    del ws_h

    if rank != 0:
        return None
    units = n_q * args.steps * world
    value = ranks.whole_job_rate(n_q * args.steps, world, ms)
    peak, peak_kind = peaks()
    score_bytes = n_q * wl.n_entries * IDX_BYTES           # algorithmic bytes of one score launch
    achieved = score_bytes / (score_ms / 1e3) / 1e9
    step_bytes = n_q * (wl.n_entries * IDX_BYTES + FIXED_BYTES_PER_QUERY)
    # csa2_decode: indexer, selection (one CTA per row; or the collection pass,
    # preceded by the maxima pass unless the supergroups are the epilogue's
    # 512-entry units or 32-entry groups), attention kernel + split merge
    def topk_launches(n):
        if n <= 16384:
            return 1
        sgi = 512
        while sgi > 8 and n // sgi < 4 * 512:
            sgi //= 2
        while -(-n // sgi) > 16384:
            sgi *= 2
        return 1 if sgi in (512, 32) else 2
    launches_per_step = 1 + topk_launches(n_max) + 2
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e2m1xe2m1->f32 (score), f16xf16 + bf16xbf16->f32 (attention)",
        "data": "synthetic (seeded counter-based generator; no trained weights)",
        "config": {"workload": wl.name, "n_seq": wl.n_seq, "n_entries": wl.n_entries, "queries_per_step": n_q,
                   "zipf_keys": wl.zipf, "topk": 512, "swa": 128, "heads": 64, "latent": 512,
                   "l2": "inputs larger than L2 (%.0f MB streamed per step)" % (step_bytes / 1e6),
                   "parallelism": f"replicas x{world} (independent batches)"},
        "path_hbm_gbs": step_bytes / (ms / args.steps / 1e3) / 1e9,
        "path_frac_of_measured_peak": step_bytes / (ms / args.steps / 1e3) / 1e9 / peak,
        "roofline": {"kernel": "index_score", "bound": "hbm", "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": INDEX_SCORE_TRAFFIC.get(wl.name),
                     "algorithmic_bytes_per_launch": score_bytes, "avg_launch_ms": score_ms,
                     "measured_in": "the indexer launch inside K further csa2_decode steps, between the "
                                    "events csa2_profile_events has it record (the step's own kernel, "
                                    "maxima included; 570.4 MB of keys per launch counted)"},
        "clocks": clk,
        "e2e": {"value": units / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "call": "csa2_decode_host on pinned host buffers (per step: the inputs read in place by one "
                        "staging grid that packs the indexer query, the decode, the output written by its last "
                        "grid into the pinned host buffer)"},
        "gpu_launches": launches_per_step * args.steps,
        "impl": "ours",
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    return line


def profiled_indexer_ms(steps, stream, step):
    """Average duration of the indexer launch inside `steps` decode steps, from
    the events csa2_profile_events has csa2_decode / csa2_decode_reindex record
    around it (recording between the step's kernels keeps the selection from
    starting early beside it: these steps are not the timed ones)."""
    import torch
    import compressed_sparse_attention_index_gb300 as C
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:                                  # (the events exist once recorded)
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    try:
        for a, b in ev:
            C.csa2_profile_events(a, b)
            step()
    finally:
        C.csa2_profile_events(None, None)
    torch.cuda.synchronize()
    assert C.csa2_get_device_status() == 0
    return sum(a.elapsed_time(b) for a, b in ev) / steps


def run_rows(args, rank, world, local_rank, wl):
    """Reindex decode (pool given) or m=2 prefill: event-timed steps, the
    dominant kernel's roofline, and the step through pinned host inputs."""
    import torch
    import torch.distributed as dist
    import compressed_sparse_attention_index_gb300 as C
    from compressed_sparse_attention_index_gb300 import decode, ranks
    from gen.device import build_device_workload

    dw = build_device_workload(wl)
    n_q, n_max = dw.q.shape[0], dw.n_max
    buf = decode.DecodeBuffers(n_q, n_max, pool=wl.pool, out_dtype=C.CSA2_OUT_BF16)
    stream = torch.cuda.current_stream()
    if wl.pool:
        decode.reindex_decode(dw, buf, None, stream, build_pool=True)     # the pool the step is given

        def step():
            decode.fused_reindex_decode(dw, buf, None, stream)
    else:
        def step():
            decode.fused_decode(dw, buf, None, stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert C.csa2_get_device_status() == 0
    clocks = ClockSampler(local_rank)
    time.sleep(0.3)
    ranks.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ranks.barrier()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    assert C.csa2_get_device_status() == 0

    # the dominant kernel: the pool-mode indexer inside K further
    # csa2_decode_reindex steps (the library's profile events around it), or
    # the prefill's attention alone in K further launches between events
    if wl.pool:
        k_ms = profiled_indexer_ms(args.steps, stream, step)
    else:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.steps):
            ev[i][0].record(stream)
            decode.attend(dw, buf, None, stream)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        k_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    assert C.csa2_get_device_status() == 0
    ms = ranks.max_over_ranks(ms, device="cuda")

    # the step through pinned host inputs: the attention query and the indexer
    # inputs of the step in, the output back
    import numpy as np
    from gen import inputs as G
    w_dev = dw.w_re if wl.pool else dw.w
    s_qidx = G.S_QIDX_RE if wl.pool else G.S_QIDX
    qidx_bits = np.concatenate([G.normal_block_bf16(wl.seed, s_qidx, qi, 0, 32, 128) for qi in range(n_q)])
    stage_h, stage_d, (q_v, w_v, qidx_v) = staged_inputs(
        [dw.q.cpu(), w_dev.cpu(), torch.from_numpy(qidx_bits.view(np.int16)).view(torch.bfloat16)])
    dw.q = q_v
    if wl.pool:
        dw.w_re = w_v
    else:
        dw.w = w_v
    out_h = torch.empty(buf.out.shape, dtype=buf.out.dtype).pin_memory()
    nib, scl = (dw.q_nib_re, dw.q_scale_re) if wl.pool else (dw.q_nib, dw.q_scale)

    def e2e_step():
        stage_d.copy_(stage_h, non_blocking=True)
        C.csa2_fp4_pack(C.CSA2_IDX_MXFP4, qidx_v, n_q * 32, 1, None, nib, scl)
        step()
        out_h.copy_(buf.out, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = ranks.max_over_ranks(e0.elapsed_time(e1), device="cuda")
    h2d = stage_h.numel()
    d2h = out_h.numel() * out_h.element_size()
    if rank != 0:
        return None

    peaks_all = {}
    pf = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pf):
        with open(pf) as f:
            peaks_all = json.load(f)
    units = n_q * args.steps * world
    n_vis = dw.n_vis.cpu().numpy().astype(np.int64)
    swa_cnt = dw.swa_cnt.cpu().numpy().astype(np.int64)
    if wl.pool:
        # pool keys + block ids + the fixed per-query bytes
        step_bytes = n_q * (16384 * IDX_BYTES + 2048 * 4 + FIXED_BYTES_PER_QUERY)
        k_bytes = n_q * 16384 * IDX_BYTES
        hbm, hbm_kind = peaks()
        roof = {"kernel": "index_score (pool mode)", "bound": "hbm", "achieved": k_bytes / (k_ms / 1e3) / 1e9,
                "peak": hbm, "peak_kind": hbm_kind, "unit": "GB/s",
                "frac": k_bytes / (k_ms / 1e3) / 1e9 / hbm, "traffic": INDEX_SCORE_TRAFFIC.get(wl.name),
                "algorithmic_bytes_per_launch": k_bytes, "avg_launch_ms": k_ms,
                "measured_in": "the pool-mode indexer launch inside K further csa2_decode_reindex steps, between "
                               "the events csa2_profile_events has it record"}
        dtype = "e2m1xe2m1->f32 (score), f16xf16 + bf16xbf16->f32 (attention)"
    else:
        # (query, entry) pairs of the attention, 4 FLOP per pair, head and dim (QK and PV)
        pairs = int(np.minimum(512, n_vis).sum() + swa_cnt.sum())
        flop = pairs * 64 * 512 * 4
        bf16 = float(peaks_all.get("bf16_tflops", 1900.0))
        achieved = flop / (k_ms / 1e3) / 1e12
        step_bytes = n_q * (65536 * 2 + 2176 + 128) + wl.n_entries * (288 + IDX_BYTES) + wl.swa_cap * 528
        roof = {"kernel": "sparse_attn", "bound": "tensor", "achieved": achieved, "peak": bf16,
                "peak_kind": "measured" if "bf16_tflops" in peaks_all else "fallback", "unit": "TFLOP/s",
                "frac": achieved / bf16, "traffic": None, "algorithmic_flop_per_launch": flop,
                "avg_launch_ms": k_ms}
        dtype = "e2m1xe2m1->f32 (score), f16xf16 + bf16xbf16->f32 (attention)"
    launches = (1 + 1 + 2) if wl.pool else (1 + 1 + 1)
    return {
        "metric": ("Reindex decode" if wl.pool else "m=2 prefill") + " query-tokens/s for CSA2 (score+top512+attn)",
        "value": units / (ms / 1e3), "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype, "data": "synthetic (seeded counter-based generator; no trained weights)",
        "config": {"workload": wl.name, "n_seq": wl.n_seq, "n_entries": wl.n_entries, "queries_per_step": n_q,
                   "m": wl.m, "pool_given": bool(wl.pool), "topk": 512, "swa": 128, "heads": 64, "latent": 512,
                   "parallelism": f"replicas x{world} (independent batches)"},
        "path_hbm_gbs": step_bytes / (ms / args.steps / 1e3) / 1e9,
        "path_frac_of_measured_peak": (step_bytes / (ms / args.steps / 1e3) / 1e9 / peaks()[0]) if wl.pool else None,
        "roofline": roof, "clocks": clk,
        "e2e": {"value": units / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches * args.steps,
        "impl": "ours",
    }


def run_mq(args, rank, world, local_rank):
    """Multi-query decode: five draft positions per sequence over the 8 x 1M
    Zipf caches, decoded in one csa2_decode_mq step; the indexer reads each
    sequence's keys once for its five queries."""
    import torch
    import compressed_sparse_attention_index_gb300 as C
    from compressed_sparse_attention_index_gb300 import decode, ranks
    from gen.device import build_device_workload
    from gen.workloads import MQ_DECODE
    wl = MQ_DECODE
    dw = build_device_workload(wl)
    n_q, n_max, G = dw.q.shape[0], dw.n_max, wl.q_per_seq
    buf = decode.DecodeBuffers(n_q, n_max, out_dtype=C.CSA2_OUT_BF16, q_group=G)
    stream = torch.cuda.current_stream()

    def step():
        decode.mq_decode(dw, buf, None, stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert C.csa2_get_device_status() == 0
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = ranks.max_over_ranks(t0.elapsed_time(t1), device="cuda")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        ev[i][0].record(stream)
        C.csa2_index_score_mq(dw.key_nib, dw.key_scale, n_max, dw.kv.shape[0], dw.q_nib, dw.q_scale, dw.w, dw.q_seq,
                              dw.n_vis, n_q, G, buf.scores, n_max, None, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    k_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    assert C.csa2_get_device_status() == 0
    if rank != 0:
        return None
    peak, peak_kind = peaks()
    key_bytes = wl.n_seq * wl.n_entries * IDX_BYTES
    step_bytes = key_bytes + n_q * FIXED_BYTES_PER_QUERY
    return {"metric": "multi-query decode query-tokens/s (5 draft positions per sequence, keys scored once per "
                      "sequence)", "value": n_q * args.steps * world / (ms / 1e3), "unit": UNIT,
            "ms_per_step": ms / args.steps, "steps": args.steps, "warmup": args.warmup,
            "queries_per_step": n_q, "key_bytes_per_step": key_bytes,
            "key_bytes_per_step_single_query_decode": wl.n_seq * wl.n_entries * IDX_BYTES,
            "path_hbm_gbs": step_bytes / (ms / args.steps / 1e3) / 1e9,
            "roofline": {"kernel": "index_score_mq (N = 160)", "bound": "hbm",
                         "achieved": key_bytes / (k_ms / 1e3) / 1e9, "peak": peak, "peak_kind": peak_kind,
                         "unit": "GB/s", "frac": key_bytes / (k_ms / 1e3) / 1e9 / peak, "traffic": None,
                         "algorithmic_bytes_per_launch": key_bytes, "avg_launch_ms": k_ms},
            "gpu_launches": 4 * args.steps}


def run_layers(args, rank, world, local_rank):
    """The decoder's twenty layers for one token of each sequence (one Full
    layer, four Reindex layers, fifteen Reuse layers borrowing selections)
    over the 8 x 1M Zipf caches, chained through the C ABI."""
    import torch
    import compressed_sparse_attention_index_gb300 as C
    from compressed_sparse_attention_index_gb300 import decode, ranks
    from gen.device import build_device_workload, build_decoder_layers
    from gen.workloads import CONFIGS, DECODER_LAYERS
    wl = CONFIGS[4]
    dw = build_device_workload(wl)
    dl = build_decoder_layers(wl, dw, DECODER_LAYERS)
    n_q = dw.q.shape[0]
    step = decode.DecoderStep(n_q, dw.n_max, DECODER_LAYERS, out_dtype=C.CSA2_OUT_BF16)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step.run(dw, dl, None, stream)
    torch.cuda.synchronize()
    assert C.csa2_get_device_status() == 0
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step.run(dw, dl, None, stream)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = ranks.max_over_ranks(t0.elapsed_time(t1), device="cuda")
    assert C.csa2_get_device_status() == 0
    if rank != 0:
        return None
    n_re = sum(1 for role, _ in DECODER_LAYERS if role == "reindex")
    n_ru = sum(1 for role, _ in DECODER_LAYERS if role == "reuse")
    return {"metric": "decoder-step query-tokens/s (20 layers: 1 Full, 4 Reindex, 15 Reuse)",
            "value": n_q * args.steps * world / (ms / 1e3), "unit": UNIT, "ms_per_step": ms / args.steps,
            "steps": args.steps, "warmup": args.warmup, "layers": len(DECODER_LAYERS),
            "layer_mix": {"full": 1, "reindex": n_re, "reuse": n_ru},
            "gpu_launches": args.steps * (4 + n_re * 2 + len(DECODER_LAYERS) * 2)}


def run_build(args, rank, world, local_rank):
    """The cache a 1,048,576-token encoder prompt leaves (m = 2: 524,288 entries):
    csa2_build_cache from bf16 tokens and fp32 gate logits in HBM to the main-cache
    records and the indexer keys' records; and the key projection alone
    (csa2_index_key_proj over the pooled latents), the tensor-core kernel of the
    build."""
    import torch
    import compressed_sparse_attention_index_gb300 as C
    from compressed_sparse_attention_index_gb300 import ranks
    n_tok, m = 1 << 20, 2
    n_e = n_tok // m
    g = torch.Generator(device="cuda").manual_seed(91 + rank)
    toks = torch.randn((n_tok, 512), generator=g, device="cuda").to(torch.bfloat16)
    z = torch.randn((n_tok, 512), generator=g, device="cuda")
    w = (torch.randn((128, 512), generator=g, device="cuda") / 512 ** 0.5).to(torch.bfloat16)
    kv = torch.empty((n_e, 288), dtype=torch.uint8, device="cuda")
    nib = torch.empty((n_e, 64), dtype=torch.uint8, device="cuda")
    sc = torch.empty((n_e, 4), dtype=torch.uint8, device="cuda")
    wsb = C.csa2_workspace_size(C.CSA2_OP_BUILD_CACHE, 0, n_tok, m)
    ws = torch.empty((wsb,), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        C.csa2_build_cache(toks, n_tok, m, z, w, kv, nib, sc, ws, wsb, stream)
    steps = max(3, min(args.steps, 20))
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert C.csa2_get_device_status() == 0
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = ranks.max_over_ranks(t0.elapsed_time(t1), device="cuda") / steps
    # the projection alone over the prompt's pooled latents (here: its first n_e tokens)
    lat = toks[:n_e]
    keys = torch.empty((n_e, 128), dtype=torch.bfloat16, device="cuda")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        C.csa2_index_key_proj(lat, n_e, w, keys, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    p_ms = sum(a.elapsed_time(b) for a, b in ev) / steps
    assert C.csa2_get_device_status() == 0
    if rank != 0:
        return None
    peak, peak_kind = peaks()
    io_bytes = n_tok * (512 * 2 + 512 * 4) + n_e * (288 + 68)          # tokens + gates in, records out
    p_bytes = n_e * (512 * 2 + 128 * 2)                                  # latents in, bf16 keys out
    return {"metric": "cache-build prompt tokens/s (1,048,576-token encoder prompt, m = 2: pooling, main-cache "
                      "records, 512 -> 128 key projection, key records)",
            "value": n_tok * world / (ms / 1e3), "unit": "prompt-tokens/s", "ms_per_step": ms, "steps": steps,
            "warmup": args.warmup, "io_bytes_per_step": io_bytes,
            "path_hbm_gbs": io_bytes / (ms / 1e3) / 1e9, "path_frac_of_measured_peak": io_bytes / (ms / 1e3) / 1e9 / peak,
            "roofline": {"kernel": "proj_keys (csa2_index_key_proj)", "bound": "hbm",
                         "achieved": p_bytes / (p_ms / 1e3) / 1e9, "peak": peak, "peak_kind": peak_kind,
                         "unit": "GB/s", "frac": p_bytes / (p_ms / 1e3) / 1e9 / peak, "traffic": None,
                         "algorithmic_bytes_per_launch": p_bytes, "avg_launch_ms": p_ms,
                         "tflops": 2.0 * n_e * 128 * 512 / (p_ms / 1e3) / 1e12},
            "gpu_launches": steps * 3 * ((n_e + 131071) // 131072)}


def run_reference(args):
    from gen.workloads import CONFIGS
    import oracle
    oracle.build()
    wl = workload_of(args)
    for _ in range(args.warmup):
        pass                       # the oracle has no state to warm; its packed keys are built once below
    t_total = 0.0
    for i in range(args.steps):
        t_total += oracle_decode_sample(wl, qi=i % wl.n_q if wl.n_q <= 1 else 0)
    per_q = t_total / args.steps
    value = 1.0 / per_q
    cores = int(os.environ.get("OMP_NUM_THREADS", cpu_cores()))
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_q * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "n_seq": wl.n_seq, "n_entries": wl.n_entries,
                   "queries_per_step": 1, "sample": "one query of sequence 0 per step"},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"one query (sequence 0) per step, full {wl.n_entries}-entry cache"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)))
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    if args.only is not None:
        r = {"mq": run_mq, "layers": run_layers, "build": run_build}[args.only](args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(r))
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    line = run_ours(args, rank, world, local_rank)
    if args.config == 4 and not args.no_extra:
        # secondary workloads in the same run, as keys of the one line: the
        # 32 x 65,536-entry decode batch and the 64 x 1,048,576 Reindex step
        import copy
        extra = {}
        for c in (1, 3):
            a2 = copy.copy(args)
            a2.config, a2.no_cpu_baseline = c, True
            a2.steps = max(3, min(args.steps, 50))
            r = run_ours(a2, rank, world, local_rank)
            if rank == 0:
                extra[r["config"]["workload"]] = {
                    k: r[k] for k in ("metric", "value", "unit", "ms_per_step", "path_hbm_gbs", "roofline", "e2e",
                                      "clocks", "gpu_launches", "steps", "warmup")
                    if k in r}
                if "path_frac_of_measured_peak" in r:
                    extra[r["config"]["workload"]]["path_frac_of_measured_peak"] = r["path_frac_of_measured_peak"]
            import torch
            torch.cuda.empty_cache()
        a2 = copy.copy(args)
        a2.steps = max(3, min(args.steps, 50))
        r = run_mq(a2, rank, world, local_rank)
        if rank == 0:
            extra["mq_decode_N1M_B8_G5_zipf"] = r
        torch.cuda.empty_cache()
        r = run_layers(a2, rank, world, local_rank)
        if rank == 0:
            extra["decoder_step_N1M_B8_zipf_20layers"] = r
        torch.cuda.empty_cache()
        r = run_build(a2, rank, world, local_rank)
        if rank == 0:
            extra["cache_build_prompt_1M_m2"] = r
        if rank == 0:
            line["secondary"] = extra
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
