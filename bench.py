"""Benchmark of the split-stream KV hot path on GB300.

One step = every row of the path on synthetic data resident in HBM:
  encode        Qwen3-235B-A22B-shaped KV at 128K: 94 layers x (K, V) =
                B 188, L 131072, 4 KV heads, D 128, page 256, C 64, alpha 255
                (23.5 GiB BF16), the largest configuration on one GPU
  decode_anchor the same streams -> BF16 KV
  decode_full   the same streams -> BF16 KV
  attn_draft    8 sequences x 32768 tokens, 32 query heads / 8 KV heads,
                T = 1 over the Anchor codes (+ split combine)
  attn_verify   the same KV, T = 8 over Anchor + Residual (+ split combine)
Metric: BF16-equivalent KV GB/s over the whole step (2 bytes per KV element
each row touches), with per-row times, roofline fractions of the measured HBM
bandwidth, and decode-attention tokens/s.  The other codec configurations
(the tiny case in microseconds, Llama-3-8B and Qwen-32B at 16K) are timed as
rows of their own under `configs`.  Sampled page blocks and attention rows of
the timed workload are compared with the CPU oracle outside the timed region
(`parity`).

Flags: --gpus N (one replica per rank under torchrun; weak scaling),
--steps K, --warmup W, --impl {lynx,reference}.  --impl reference times the
CPU oracle (the only reference this path has): each step is one fixed sample
of the same rows.  Profiling aids: --rows a,b selects rows; --small shrinks
both workloads (codec B = 8, attention batch 2; still larger than L2) and
skips the e2e, parity, extras and CPU legs; --codec NAME times another codec
configuration as the step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV codec GB/s (BF16-equivalent) and anchor-attention tokens/s; % of HBM roofline"
ALPHA = 255.0
# The codec configurations: B = 2 x layers (K and V interleaved), L tokens,
# H KV heads, D channels, page P, chunk C.
CODEC_CONFIGS = {
    "tiny": dict(B=2, L=256, H=1, D=128, P=256, C=32, n_outlier=2),
    "llama3-8b-16k": dict(B=64, L=16384, H=8, D=128, P=128, C=32),
    "qwen-32b-16k": dict(B=128, L=16384, H=8, D=128, P=128, C=32),
    "qwen3-235b-128k": dict(B=188, L=131072, H=4, D=128, P=256, C=64),
}
HEADLINE = "qwen3-235b-128k"
# the widened rows (variants, split stream) run on this configuration
EXTRAS_CODEC = "llama3-8b-16k"
CODEC = dict(CODEC_CONFIGS[HEADLINE], name=HEADLINE)
ATTN = dict(batch=8, L=32768, H_kv=8, H_q=32, D=128, P=128, C=32, T_draft=1, T_verify=8)
# the tiny configuration's attention: 1 KV head, 1 query head, 256 tokens
TINY_ATTN = dict(batch=1, L=256, H_kv=1, H_q=1, D=128, P=256, C=32, T_draft=1, T_verify=8,
                 n_outlier=2)


def meta_bytes_per_elem(P, C):
    return 8.0 / P + 8.0 / C


def codec_elems(c=None):
    c = c or CODEC
    return c["B"] * c["L"] * c["H"] * c["D"]


def attn_kv_elems(a=None):
    a = a or ATTN
    return 2 * a["batch"] * a["L"] * a["H_kv"] * a["D"]   # K and V


def codec_bytes(c=None):
    """Bytes each codec row must move at minimum (per launch)."""
    c = c or CODEC
    n = codec_elems(c)
    m = meta_bytes_per_elem(c["P"], c["C"])
    return {"encode": n * (2 + 0.5 + 0.5 + m),
            "decode_anchor": n * (0.5 + m + 2),
            "decode_full": n * (0.5 + 0.5 + m + 2)}


def attn_bytes(a=None):
    """Bytes each attention row must read at minimum (per launch): the packed
    K and V (q and the output are a few hundred KB)."""
    a = a or ATTN
    na = attn_kv_elems(a)
    ma = meta_bytes_per_elem(a["P"], a["C"])
    return {"attn_draft": na * (0.5 + ma), "attn_verify": na * (1.0 + ma)}


def algorithmic_bytes():
    """Bytes each row of the step must move at minimum (per launch)."""
    return {**codec_bytes(), **attn_bytes()}


def bf16_equiv_bytes(c=None, a=None):
    n = codec_elems(c)
    na = attn_kv_elems(a)
    return {"encode": 2 * n, "decode_anchor": 2 * n, "decode_full": 2 * n,
            "attn_draft": 2 * na, "attn_verify": 2 * na}


ROWS = ["encode", "decode_anchor", "decode_full", "attn_draft", "attn_verify"]
CODEC_ROWS = ROWS[:3]
ATTN_ROWS = ROWS[3:]
# kernel launches of one call of each row
LAUNCHES = {"encode": 1, "decode_anchor": 1, "decode_full": 1, "attn_draft": 2,
            "attn_verify": 2}


# Sources that define each row's kernel; the recorded DRAM traffic of a
# kernel is only reported while these files are unchanged.
ROW_SOURCES = {
    "encode": ["encode.cu", "common.cuh", "internal.h"],
    "decode_anchor": ["decode.cu", "common.cuh", "internal.h"],
    "decode_full": ["decode.cu", "common.cuh", "internal.h"],
    "attn_draft": ["attn.cu", "attn_params.h", "common.cuh", "internal.h"],
    "attn_verify": ["attn_tc.cu", "attn.cu", "attn_params.h", "common.cuh", "internal.h"],
}
TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


def sources_hash(row):
    import hashlib
    h = hashlib.sha256()
    for name in ROW_SOURCES[row]:
        with open(os.path.join(ROOT, "split_stream_kv_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_records():
    if not os.path.exists(TRAFFIC):
        return {}
    with open(TRAFFIC) as f:
        return json.load(f).get("rows", {})


def recorded_traffic(row, units_per_launch, config=None):
    """DRAM bytes per launch of the row's kernel, scaled by the units it
    processes from the ncu capture recorded in profiles/traffic.json, or None
    if there is no record of this row's kernel on this configuration for the
    current sources."""
    rec = traffic_records().get(row)
    if not rec:
        return None
    if rec.get("sources") != sources_hash(row):
        return None
    want = config or (CODEC["name"] if row in CODEC_ROWS else "attention-32k")
    if rec.get("config") != want:
        return None
    return int(round(float(rec["dram_bytes"]) / float(rec["units"]) * units_per_launch))


def units_per_launch(row):
    """Elements (KV elements read or written) one launch of the row handles."""
    return codec_elems() if row in CODEC_ROWS else attn_kv_elems()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def codec_desc(name, c):
    return (f"{name}-shaped KV codec (B={c['B']} = {c['B'] // 2} layers x K,V; L={c['L']}; "
            f"H_kv={c['H']}; D={c['D']}; page={c['P']}; C={c['C']}; alpha={ALPHA:g})")


def workload_config():
    gib = codec_elems() * 2 / 2 ** 30
    return {
        "workload": (codec_desc(CODEC["name"], CODEC) + " + packed-KV decode attention "
                     f"({ATTN['batch']} seqs x {ATTN['L']} tokens; H_q={ATTN['H_q']} over "
                     f"H_kv={ATTN['H_kv']}; page={ATTN['P']}; C={ATTN['C']}; draft T=1 "
                     "anchor, verify T=8 full)"),
        "l2": (f"inputs larger than L2 ({gib:.1f} GiB BF16 codec input, "
               f"{attn_bytes()['attn_verify'] / 2 ** 30:.2f} GiB packed attention KV)"),
        "parallelism": "replicas",
    }


def slices_of(B, most=8):
    """Largest slice count <= most that divides B (the e2e leg's pipeline)."""
    for n in range(most, 0, -1):
        if B % n == 0:
            return n
    return 1


# ----------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.proc = None
        self.path = None
        if not uuid:
            return
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", uuid, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx.append(float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------- CPU leg

class CpuSample:
    """A fixed sample of the step for the CPU oracle: page blocks of the
    headline codec (encode and both decodes of 2 x Lc tokens x its heads)
    and attention of one (sequence, KV head) pair over La tokens (both
    decoders of its pages, then the float64 softmax for the 4 draft rows and
    the 32 verify rows)."""

    def __init__(self, Lc=4096, La=4096):
        import numpy as np
        import torch

        import oracle
        from split_stream_kv_gb300 import synth
        oracle.build()
        c, a = CODEC, ATTN
        self.Lc, self.La = Lc, La
        kv = synth.kv_cache(2, Lc, c["H"], 128, seed=11, device="cpu")
        self.bits = kv.view(torch.int16).numpy().view(np.uint16)
        kva = synth.kv_cache(2, La, 1, 128, seed=5, device="cpu")
        ab = kva.view(torch.int16).numpy().view(np.uint16)
        self.enc = oracle.encode(ab, a["P"], a["C"], ALPHA)
        self.q = np.random.default_rng(0).standard_normal(
            (a["T_verify"] * (a["H_q"] // a["H_kv"]), 128)).astype(np.float32)

    def desc(self):
        c = CODEC
        return (f"{2 * (self.Lc // c['P']) * c['H']} page blocks of the {c['name']} codec "
                f"(2 x {self.Lc} tokens x {c['H']} heads) encoded and decoded both ways + "
                f"draft (4 rows) and verify (32 rows) attention over one {self.La}-token "
                f"(sequence, KV head) pair incl. its decode")

    def run(self, threads):
        """One pass: (codec seconds, codec BF16 bytes, attention seconds,
        attention BF16 bytes)."""
        import oracle
        c, a = CODEC, ATTN
        t0 = time.perf_counter()
        oa, orr, om = oracle.encode(self.bits, c["P"], c["C"], ALPHA, threads=threads)
        oracle.decode(oa, None, om, self.Lc, c["P"], c["C"], ALPHA, threads=threads)
        oracle.decode(oa, orr, om, self.Lc, c["P"], c["C"], ALPHA, threads=threads)
        t_codec = time.perf_counter() - t0
        t0 = time.perf_counter()
        ea, er, em = self.enc
        G = a["H_q"] // a["H_kv"]
        for full, rows in ((False, G * a["T_draft"]), (True, G * a["T_verify"])):
            x = oracle.decode(ea, er if full else None, em, self.La, a["P"], a["C"], ALPHA,
                              threads=threads)
            xb = oracle.bf16_bits_to_f32(oracle.f32_to_bf16_bits(x)).reshape(x.shape)
            K, V = xb[0, :, 0], xb[1, :, 0]
            for r in range(rows):
                oracle.attention_row(self.q[r], K, V)
        t_attn = time.perf_counter() - t0
        return t_codec, 3 * 2 * self.bits.size, t_attn, 2 * 2 * 2 * self.La * 128


def step_rate(t_codec, codec_b, t_attn, attn_b):
    """GB/s BF16-equivalent of the step's byte mix from the sample's codec and
    attention rates (each reweighted to the step's share of bytes)."""
    be = bf16_equiv_bytes()
    w_codec = be["encode"] + be["decode_anchor"] + be["decode_full"]
    w_attn = be["attn_draft"] + be["attn_verify"]
    t_step = w_codec / (codec_b / t_codec) + w_attn / (attn_b / t_attn)
    return (w_codec + w_attn) / t_step / 1e9


def cpu_sample_run(target_s: float = 12.0, threads: int | None = None, sample=None):
    """Time the oracle on the fixed sample, repeated until about target_s
    seconds of work.  Returns (GB/s BF16-equivalent, threads, description,
    seconds)."""
    threads = threads or (os.cpu_count() or 1)
    sample = sample or CpuSample()
    tc = ta = 0.0
    bc = ba = 0
    reps = 0
    while tc + ta < target_s or reps == 0:
        a, b, c_, d = sample.run(threads)
        tc, bc, ta, ba = tc + a, bc + b, ta + c_, ba + d
        reps += 1
    value = step_rate(tc, bc, ta, ba)
    desc = (f"{reps} x [{sample.desc()}]; {tc + ta:.1f} s on {threads} thread"
            f"{'s' if threads > 1 else ''}; codec and attention rates reweighted to the "
            "step's byte mix")
    return value, threads, desc, tc + ta


# ----------------------------------------------------------------- GPU leg

def max_over_ranks(vals, world, device=None):
    """Max of each value over all ranks (a timing reduction, not data)."""
    if world <= 1:
        return list(vals)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(vals), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_gbps(step_bytes_per_rank, world, seconds_per_step):
    """Weak scaling: every rank processes its own workload."""
    return world * step_bytes_per_rank / seconds_per_step / 1e9


def attn_setup(a, dev, seed=5):
    """Packed K and V of an attention workload, its queries, outputs and a
    workspace for both steps."""
    import torch

    from split_stream_kv_gb300 import lynx, synth
    kva = synth.kv_cache(2 * a["batch"], a["L"], a["H_kv"], a["D"], seed=seed, device=dev,
                         n_outlier=a.get("n_outlier"))
    ks = lynx.lynx_encode(kva[0::2].contiguous(), a["P"], a["C"], ALPHA)
    vs = lynx.lynx_encode(kva[1::2].contiguous(), a["P"], a["C"], ALPHA)
    del kva
    q1 = synth.queries(a["batch"], a["T_draft"], a["H_q"], a["D"], seed=1, device=dev)
    q8 = synth.queries(a["batch"], a["T_verify"], a["H_q"], a["D"], seed=8, device=dev)
    out1 = torch.empty((a["batch"], a["T_draft"], a["H_q"], a["D"]), device=dev)
    out8 = torch.empty((a["batch"], a["T_verify"], a["H_q"], a["D"]), device=dev)
    ws_n = max(lynx.lynx_attn_workspace_bytes(a["batch"], t, a["H_q"], a["L"], a["H_kv"],
                                              a["D"], a["P"])
               for t in (a["T_draft"], a["T_verify"]))
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)
    return dict(ks=ks, vs=vs, q1=q1, q8=q8, out1=out1, out8=out8, ws=ws)


def attn_row(name, a, t):
    from split_stream_kv_gb300 import lynx
    ks, vs = t["ks"], t["vs"]
    if name == "attn_draft":
        lynx.lynx_attn_decode(t["q1"], (ks[0], None, ks[2]), (vs[0], None, vs[2]), a["L"],
                              a["P"], a["C"], ALPHA, lynx.LYNX_ANCHOR, out=t["out1"],
                              workspace=t["ws"])
    else:
        lynx.lynx_attn_decode(t["q8"], ks, vs, a["L"], a["P"], a["C"], ALPHA, lynx.LYNX_FULL,
                              out=t["out8"], workspace=t["ws"])


def codec_row(name, c, t):
    from split_stream_kv_gb300 import lynx
    if name == "encode":
        lynx.lynx_encode(t["kv"], c["P"], c["C"], ALPHA, t["anc"], t["res"], t["meta"])
    elif name == "decode_anchor":
        lynx.lynx_decode_anchor(t["anc"], t["meta"], c["L"], c["P"], c["C"], ALPHA,
                                out=t["dec_a"])
    else:
        lynx.lynx_decode_full(t["anc"], t["res"], t["meta"], c["L"], c["P"], c["C"], ALPHA,
                              out=t["dec_f"])


def codec_setup(c, dev, seed=11):
    import torch

    from split_stream_kv_gb300 import lynx, synth
    kv = synth.kv_cache(c["B"], c["L"], c["H"], c["D"], seed=seed, device=dev,
                        n_outlier=c.get("n_outlier"))
    anc, res, meta = lynx.lynx_encode(kv, c["P"], c["C"], ALPHA)
    return dict(kv=kv, anc=anc, res=res, meta=meta, dec_a=torch.empty_like(kv),
                dec_f=torch.empty_like(kv))


def run_lynx(args, rank, world, dev):
    import torch

    from split_stream_kv_gb300 import lynx

    torch.cuda.set_device(dev)
    c = CODEC
    a = ATTN
    tc = codec_setup(c, dev, seed=11 + rank)
    ta = attn_setup(a, dev, seed=5 + rank)

    def row(name):
        if name in CODEC_ROWS:
            codec_row(name, c, tc)
        else:
            attn_row(name, a, ta)

    rows_run = [r for r in ROWS if r in args.rows]
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    # clocks are sampled from the warm-up on, through the timed region, and
    # over untimed repeats of the same step until about 2 s of samples exist
    clocks = ClockSampler(uuid if rank == 0 else None)
    t_clock0 = time.perf_counter()
    for _ in range(args.warmup):
        for r in rows_run:
            row(r)
    torch.cuda.synchronize(dev)

    # ---- device-timed region
    ev = {r: [] for r in rows_run}
    barrier()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        for r in rows_run:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            row(r)
            e1.record(stream)
            ev[r].append((e0, e1))
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    while time.perf_counter() - t_clock0 < 2.0:
        for r in rows_run:
            row(r)
        torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms_total = t_start.elapsed_time(t_end)
    row_ms = {r: sum(e0.elapsed_time(e1) for e0, e1 in ev[r]) / args.steps for r in rows_run}
    launches = sum(LAUNCHES[r] for r in rows_run) * args.steps
    if args.small or rows_run != ROWS:
        ms_total, = max_over_ranks([ms_total], world, dev)
        return dict(ms_total=ms_total, row_ms=row_ms, e2e_s=None, h2d=0, d2h=0, clocks=clk,
                    launches=launches)

    e2e_s, h2d, d2h = run_e2e(args, tc, ta, dev, barrier)
    ms_total, e2e_s = max_over_ranks([ms_total, e2e_s], world, dev)
    parity = extras = configs = None
    if rank == 0:
        parity = {"codec": codec_parity(c, tc, dev), "attention": attn_parity(a, ta, dev)}
    assert lynx.lynx_wait_timeouts() == 0
    del tc
    torch.cuda.empty_cache()
    if rank == 0:
        configs = measure_configs(dev)
        extras = measure_all_extras(ta, dev, rank)
    assert lynx.lynx_wait_timeouts() == 0
    return dict(ms_total=ms_total, row_ms=row_ms, e2e_s=e2e_s, h2d=h2d, d2h=d2h, clocks=clk,
                launches=launches, extras=extras, configs=configs, parity=parity)


def run_e2e(args, tc, ta, dev, barrier):
    """The same step end to end through the public API: every step copies its
    inputs in from pinned host buffers and its results (code streams and
    attention outputs) back.  Returns (seconds per step, bytes in, bytes out
    per step)."""
    import torch

    from split_stream_kv_gb300 import lynx
    c, a = CODEC, ATTN
    kv, anc, res, meta = tc["kv"], tc["anc"], tc["res"], tc["meta"]
    dec_a, dec_f = tc["dec_a"], tc["dec_f"]
    ks, vs, q1, q8 = ta["ks"], ta["vs"], ta["q1"], ta["q8"]
    out1, out8, ws = ta["out1"], ta["out8"], ta["ws"]
    kv_h = torch.empty(kv.shape, dtype=kv.dtype, pin_memory=True)
    kv_h.copy_(kv)
    pk_h = [t.cpu().pin_memory() for t in (ks[0], ks[1], ks[2], vs[0], vs[1], vs[2])]
    pk_d = [torch.empty_like(t, device=dev) for t in pk_h]
    q1_h, q8_h = q1.cpu().pin_memory(), q8.cpu().pin_memory()
    anc_h = torch.empty(anc.shape, dtype=anc.dtype, pin_memory=True)
    res_h = torch.empty(res.shape, dtype=res.dtype, pin_memory=True)
    meta_h = torch.empty(meta.shape, dtype=meta.dtype, pin_memory=True)
    o1_h = torch.empty(out1.shape, dtype=out1.dtype, pin_memory=True)
    o8_h = torch.empty(out8.shape, dtype=out8.dtype, pin_memory=True)
    h2d = kv_h.nbytes + sum(t.nbytes for t in pk_h) + q1_h.nbytes + q8_h.nbytes
    d2h = anc_h.nbytes + res_h.nbytes + meta_h.nbytes + o1_h.nbytes + o8_h.nbytes

    # The step is pipelined over three streams, as the pages' serializer
    # overlaps the transfer of one page with the quantisation of the next:
    # the BF16 input arrives in slices and each slice is encoded as soon as
    # it has landed; the code streams of a slice go back to the host while
    # later slices are encoded and the decoders and attention run.  Events
    # keep the reuse of the device buffers across steps ordered.
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    nsl = slices_of(c["B"])
    bs = c["B"] // nsl
    ev_in = [torch.cuda.Event() for _ in range(nsl)]
    ev_enc = [torch.cuda.Event() for _ in range(nsl)]
    ev_back = [torch.cuda.Event() for _ in range(nsl)]
    ev_attn_in, ev_cmp, ev_res_back = (torch.cuda.Event() for _ in range(3))
    first = [True]

    def e2e_step():
        for k in range(nsl):
            sl = slice(k * bs, (k + 1) * bs)
            with torch.cuda.stream(s_in):
                if not first[0]:
                    s_in.wait_event(ev_enc[k])        # last step's encode has read kv[sl]
                kv[sl].copy_(kv_h[sl], non_blocking=True)
                ev_in[k].record(s_in)
        with torch.cuda.stream(s_in):
            if not first[0]:
                s_in.wait_event(ev_cmp)               # last step's attention is done
            for d, hsrc in zip(pk_d, pk_h):
                d.copy_(hsrc, non_blocking=True)
            q1.copy_(q1_h, non_blocking=True)
            q8.copy_(q8_h, non_blocking=True)
            ev_attn_in.record(s_in)
        with torch.cuda.stream(s_cmp):
            for k in range(nsl):
                sl = slice(k * bs, (k + 1) * bs)
                s_cmp.wait_event(ev_in[k])
                if not first[0]:
                    s_cmp.wait_event(ev_back[k])      # last step's codes of sl are home
                lynx.lynx_encode(kv[sl], c["P"], c["C"], ALPHA, anc[sl], res[sl], meta[sl])
                ev_enc[k].record(s_cmp)
            lynx.lynx_decode_anchor(anc, meta, c["L"], c["P"], c["C"], ALPHA, out=dec_a)
            lynx.lynx_decode_full(anc, res, meta, c["L"], c["P"], c["C"], ALPHA, out=dec_f)
            s_cmp.wait_event(ev_attn_in)
            if not first[0]:
                s_cmp.wait_event(ev_res_back)         # last step's outputs are home
            lynx.lynx_attn_decode(q1, (pk_d[0], None, pk_d[2]), (pk_d[3], None, pk_d[5]),
                                  a["L"], a["P"], a["C"], ALPHA, lynx.LYNX_ANCHOR, out=out1,
                                  workspace=ws)
            lynx.lynx_attn_decode(q8, tuple(pk_d[0:3]), tuple(pk_d[3:6]), a["L"], a["P"],
                                  a["C"], ALPHA, lynx.LYNX_FULL, out=out8, workspace=ws)
            ev_cmp.record(s_cmp)
        with torch.cuda.stream(s_out):
            for k in range(nsl):
                sl = slice(k * bs, (k + 1) * bs)
                s_out.wait_event(ev_enc[k])
                anc_h[sl].copy_(anc[sl], non_blocking=True)
                res_h[sl].copy_(res[sl], non_blocking=True)
                meta_h[sl].copy_(meta[sl], non_blocking=True)
                ev_back[k].record(s_out)
            s_out.wait_event(ev_cmp)
            o1_h.copy_(out1, non_blocking=True)
            o8_h.copy_(out8, non_blocking=True)
            ev_res_back.record(s_out)
        first[0] = False

    e2e_step()
    torch.cuda.synchronize(dev)
    barrier()
    w0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier()
    e2e_s = (time.perf_counter() - w0) / args.steps
    del kv_h, pk_h, pk_d, anc_h, res_h, meta_h, o1_h, o8_h
    return e2e_s, h2d, d2h


# ------------------------------------------------------- parity of the step

def bits16(t):
    import numpy as np
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def codec_parity(c, tc, dev, nsamp=64, seed=123):
    """Seeded page blocks of the timed codec workload (with the first and the
    last) against the oracle, outside the timed region: differing code bytes
    of the Anchor and Residual streams, differing metadata floats, and BF16
    decoder outputs (full and Anchor-only) that differ from the oracle's
    float32 decode rounded to nearest even."""
    import numpy as np
    import torch

    import oracle
    kv, anc, res, meta = tc["kv"], tc["anc"], tc["res"], tc["meta"]
    B, L, H, P, C = c["B"], c["L"], c["H"], c["P"], c["C"]
    NB = L // P
    for name in CODEC_ROWS:          # the decoders' outputs as the step left them
        codec_row(name, c, tc)
    torch.cuda.synchronize(dev)
    rng = np.random.default_rng(seed)
    blks = np.unique(np.concatenate([[0, B * NB * H - 1], rng.integers(0, B * NB * H, nsamp)]))
    hh = torch.as_tensor(blks % H, device=dev)
    pp = torch.as_tensor((blks // H) % NB, device=dev)
    bb = torch.as_tensor(blks // (H * NB), device=dev)
    tok = pp[:, None] * P + torch.arange(P, device=dev)[None, :]
    tb = bits16(kv[bb[:, None], tok, hh[:, None]])
    ga, gr = anc[bb, pp, hh].cpu().numpy(), res[bb, pp, hh].cpu().numpy()
    gm = meta[bb, pp, hh].cpu().numpy()
    gf = bits16(tc["dec_f"][bb[:, None], tok, hh[:, None]])
    gp = bits16(tc["dec_a"][bb[:, None], tok, hh[:, None]])
    n = dict(code=0, meta=0, full=0, anchor=0)
    for i in range(len(blks)):
        oa, orr, om = oracle.encode_block(tb[i], C, ALPHA)
        n["code"] += int((ga[i] != oa).sum() + (gr[i] != orr).sum())
        n["meta"] += int((gm[i].view(np.uint32) != om.view(np.uint32)).sum())
        rf = oracle.f32_to_bf16_bits(oracle.decode_block(oa, orr, om, C, ALPHA))
        rp = oracle.f32_to_bf16_bits(oracle.decode_block(oa, None, om, C, ALPHA))
        n["full"] += int((gf[i] != rf).sum())
        n["anchor"] += int((gp[i] != rp).sum())
    elems = len(blks) * P * c["D"]
    return {"blocks": int(len(blks)), "elements": int(elems),
            "code_byte_mismatches": n["code"], "meta_mismatches": n["meta"],
            "decode_full_bf16_mismatches": n["full"],
            "decode_anchor_bf16_mismatches": n["anchor"],
            "allowed_code_mismatch_fraction": 1e-6}


def attn_parity(a, ta, dev, pairs=((0, 0), (5, 3))):
    """Both attention rows of the timed workload for a few (sequence, KV head)
    pairs, against float64 oracle attention over the oracle's decode of the
    same codes rounded to BF16: the largest absolute error over all channels,
    over channels whose |V^| stays below 16 (the non-outlier channels), and
    divided by max(1, max_t |V^|) per channel (the 2e-3 acceptance)."""
    import numpy as np
    import torch

    import oracle
    for name in ATTN_ROWS:
        attn_row(name, a, ta)
    torch.cuda.synchronize(dev)
    P, C, L, G = a["P"], a["C"], a["L"], a["H_q"] // a["H_kv"]
    out = {}
    for name, T, full in (("attn_draft", a["T_draft"], False),
                          ("attn_verify", a["T_verify"], True)):
        q = (ta["q1"] if not full else ta["q8"]).float().cpu().numpy()
        o = (ta["out1"] if not full else ta["out8"]).cpu().numpy()
        worst = dict(raw=0.0, raw_small=0.0, norm=0.0)
        for b, h in pairs:
            kv_hat = []
            for s in (ta["ks"], ta["vs"]):
                an = s[0][b:b + 1, :, h:h + 1].contiguous().cpu().numpy()
                rs = s[1][b:b + 1, :, h:h + 1].contiguous().cpu().numpy() if full else None
                me = s[2][b:b + 1, :, h:h + 1].contiguous().cpu().numpy()
                x = oracle.decode(an, rs, me, L, P, C, ALPHA)[0, :, 0]
                kv_hat.append(oracle.bf16_bits_to_f32(oracle.f32_to_bf16_bits(x)).reshape(x.shape))
            K, V = kv_hat
            vmax = np.abs(V).max(axis=0)
            small = vmax < 16
            for t in range(T):
                for g in range(G):
                    ref = oracle.attention_row(q[b, t, h * G + g], K, V)
                    err = np.abs(o[b, t, h * G + g].astype(np.float64) - ref)
                    worst["raw"] = max(worst["raw"], float(err.max()))
                    worst["raw_small"] = max(worst["raw_small"], float(err[small].max()))
                    worst["norm"] = max(worst["norm"], float((err / np.maximum(1, vmax)).max()))
        out[name] = {"pairs": [list(p) for p in pairs], "rows": T * G * len(pairs),
                     "max_abs_raw": worst["raw"], "max_abs_raw_non_outlier": worst["raw_small"],
                     "max_abs_normalised": worst["norm"], "tolerance": 2e-3}
    return out


# ------------------------------------------------------ the other configs

def median_ms(fn, dev, reps, flush=None, warm=3):
    import torch
    stream = torch.cuda.current_stream(dev)
    for _ in range(warm):
        fn()
    ts = []
    for _ in range(reps):
        if flush is not None:
            flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def graph_us(fns, dev, reps=200):
    """Device latency of `fns` run in order, captured once as a CUDA graph and
    replayed `reps` times back to back between two events (so the host's
    per-call work is out of the measurement): microseconds per replay."""
    import torch
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for f in fns:
            f()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for f in fns:
            f()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) * 1e3 / reps
    del g
    return round(us, 2)


def measure_configs(dev, reps=20):
    """The codec rows on every other configuration (median of `reps` CUDA-event
    timings after 3 warm-ups, L2 flushed between repetitions), with each row's
    roofline fraction.  The tiny configuration sits in L2 and is bound by
    launch latency, so it reports microseconds (no flush), for its attention
    rows too: "us" for one call through the binding (the host's work
    included), "graph_us" per replay of the row captured as a CUDA graph, and
    "step_graph_us" for the whole tiny step (encode, both decodes, draft and
    verification) as one graph."""
    import torch
    peak, _ = load_peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    for name in ("tiny", "llama3-8b-16k", "qwen-32b-16k"):
        c = CODEC_CONFIGS[name]
        tc = codec_setup(c, dev)
        alg = codec_bytes(c)
        rows = {}
        for r in CODEC_ROWS:
            if name == "tiny":
                ms = median_ms(lambda: codec_row(r, c, tc), dev, 100)
                rows[r] = {"us": round(ms * 1e3, 2)}
            else:
                ms = median_ms(lambda: codec_row(r, c, tc), dev, reps, flush)
                ach = alg[r] / (ms / 1e3) / 1e9
                rows[r] = {"ms": round(ms, 4), "algorithmic_bytes": int(alg[r]),
                           "achieved_GBps": round(ach, 1), "roofline_frac": round(ach / peak, 4),
                           "bf16_equiv_GBps": round(2 * codec_elems(c) / (ms / 1e3) / 1e9, 1)}
        step_graph = None
        if name == "tiny":
            ta = attn_setup(TINY_ATTN, dev)
            for r in ATTN_ROWS:
                ms = median_ms(lambda: attn_row(r, TINY_ATTN, ta), dev, 100)
                rows[r] = {"us": round(ms * 1e3, 2)}
            try:
                fns = {r: (lambda r=r: codec_row(r, c, tc)) for r in CODEC_ROWS}
                fns.update({r: (lambda r=r: attn_row(r, TINY_ATTN, ta)) for r in ATTN_ROWS})
                for r, f in fns.items():
                    rows[r]["graph_us"] = graph_us([f], dev)
                step_graph = graph_us(list(fns.values()), dev)
            except Exception as ex:   # a capture the runtime refuses: say so
                step_graph = f"not captured: {type(ex).__name__}: {ex}"[:200]
            del ta
        out[name] = {"workload": codec_desc(name, c), "rows": rows}
        if step_graph is not None:
            out[name]["step_graph_us"] = step_graph
        del tc
        torch.cuda.empty_cache()
    return out


def measure_all_extras(ta, dev, rank):
    import torch

    from split_stream_kv_gb300 import synth
    a = ATTN
    c = dict(CODEC_CONFIGS[EXTRAS_CODEC], name=EXTRAS_CODEC)
    extras = measure_extras(ta["ks"], ta["vs"], ta["q8"], ta["ws"], dev)
    tc = codec_setup(c, dev, seed=11 + rank)
    kv_h = torch.empty(tc["kv"].shape, dtype=tc["kv"].dtype, pin_memory=True)
    kv_h.copy_(tc["kv"])
    host = tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                 for t in (tc["anc"], tc["res"], tc["meta"]))
    for h_, d_ in zip(host, (tc["anc"], tc["res"], tc["meta"])):
        h_.copy_(d_)
    extras["split_stream"] = measure_split(c, tc["kv"], kv_h, (tc["anc"], tc["res"], tc["meta"]),
                                           host, tc["dec_a"], dev)
    extras["variants"] = measure_variants(c, tc["kv"], tc["anc"], tc["res"], tc["meta"], dev)
    del tc, kv_h, host
    torch.cuda.empty_cache()
    kva = synth.kv_cache(4, a["L"], a["H_kv"], a["D"], seed=5 + rank, device=dev)
    qa = synth.queries(2, a["T_verify"], a["H_q"], a["D"], seed=8, device=dev)
    extras["accuracy"] = accuracy_table(kva[0::2].contiguous(), kva[1::2].contiguous(), qa,
                                        a["P"], a["C"], ALPHA)
    extras["accuracy"]["what"] = (
        "vNMSE of attention outputs (2 sequences x 32768 tokens x 8 KV heads, 8 query "
        "tokens x 32 heads) against attention over the BF16 KV; codecs on the GPU")
    return extras


def measure_extras(ks, vs, q8, ws, dev, reps=10):
    """Capabilities beyond the headline step, timed on their own with CUDA
    events (3 warm-up calls; an L2 flush between timed calls): verification
    with the draft tokens' own keys and values, verification over paged
    streams through a scattered block table, and speculative verification
    (Eq. 10-11) over a 128,256-token vocabulary."""
    import torch

    from split_stream_kv_gb300 import lynx, synth
    a = ATTN
    peak, _ = load_peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timed(fn):
        for _ in range(3):
            fn()
        ms = 0.0
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize(dev)
            ms += e0.elapsed_time(e1)
        return ms / reps

    def entry(ms, nbytes, **kw):
        ach = nbytes / (ms / 1e3) / 1e9
        return dict(ms=round(ms, 4), algorithmic_bytes=int(nbytes), achieved_GBps=round(ach, 1),
                    roofline_frac=round(ach / peak, 4), **kw)

    out = {}
    verify_bytes = attn_bytes()["attn_verify"]
    T = a["T_verify"]
    tail = synth.kv_cache(2 * a["batch"], T, a["H_kv"], a["D"], seed=77, device=dev)
    kt, vt = tail[0::2].contiguous(), tail[1::2].contiguous()
    o8 = torch.empty((a["batch"], T, a["H_q"], a["D"]), device=dev)
    ms = timed(lambda: lynx.lynx_attn_decode(q8, ks, vs, a["L"], a["P"], a["C"], ALPHA,
                                             lynx.LYNX_FULL, out=o8, workspace=ws, k_tail=kt,
                                             v_tail=vt))
    out["attn_verify_tail"] = entry(ms, verify_bytes + 2 * kt.nbytes,
                                    what=f"T={T} verification with the draft tokens' own BF16 "
                                         "keys and values (causal)")
    NB = a["L"] // a["P"]
    nblocks = a["batch"] * NB + 64
    g = torch.Generator().manual_seed(5)
    table = torch.randperm(nblocks, generator=g)[: a["batch"] * NB].view(a["batch"], NB)
    table = table.to(torch.int32).to(dev)
    idx = table.view(-1).long()

    def pool(t):  # dense [batch][NB][H][...] -> pool [nblocks][H][...] scattered by the table
        p = torch.zeros((nblocks,) + tuple(t.shape[2:]), dtype=t.dtype, device=dev)
        p[idx] = t.reshape((-1,) + tuple(t.shape[2:]))
        return p
    kp = tuple(pool(t) for t in ks)
    vp = tuple(pool(t) for t in vs)
    ms = timed(lambda: lynx.lynx_attn_decode_paged(q8, kp, vp, table, a["L"], a["P"], a["C"],
                                                   ALPHA, lynx.LYNX_FULL, out=o8, workspace=ws))
    out["attn_verify_paged"] = entry(ms, verify_bytes + table.nbytes,
                                     what=f"T={T} verification over paged streams, "
                                          f"{nblocks} physical pages behind a scattered table")
    del kp, vp
    V, B = 128256, a["batch"]
    gen = torch.Generator(device=dev).manual_seed(3)
    logits = torch.randn((B, T + 1, V), generator=gen, device=dev) * 3.0
    p = torch.softmax(logits, dim=-1)
    q = torch.softmax(logits[:, :T] + 0.05 * torch.randn((B, T, V), generator=gen, device=dev),
                      dim=-1)
    s = torch.multinomial(q.reshape(-1, V), 1, generator=gen).view(B, T).to(torch.int32)
    u = torch.rand((B, T), generator=gen, device=dev)
    r = torch.randint(-2 ** 31, 2 ** 31 - 1, (B,), generator=gen, device=dev, dtype=torch.int32)
    ms = timed(lambda: lynx.lynx_spec_verify(p, q, s, u, r))
    k, _ = lynx.lynx_spec_verify(p, q, s, u, r)
    # a sequence that rejects at k reads the rows p_k and q_k; one that accepts
    # every draft token reads p_{T+1} alone
    rows_read = int((k < T).sum()) * 2 + int((k == T).sum())
    out["spec_verify"] = entry(ms, rows_read * V * 4,
                               what=f"Eq. 10-11: batch {B}, T={T}, V={V}; mean accepted "
                                    f"{float(k.float().mean()):.2f} of {T}")
    return out


def _attention_f64(q, K, V):
    """softmax(q K^T / sqrt(D)) V in float64 on the device, for the accuracy
    table only (GQA: query head h reads KV head h // (H_q / H_kv))."""
    import torch
    B, T, Hq, D = q.shape
    Hkv = K.shape[2]
    qf = q.double().view(B, T, Hkv, Hq // Hkv, D)
    s = torch.einsum("bthgd,blhd->bhtgl", qf, K.double()) / math.sqrt(D)
    p = torch.softmax(s, dim=-1)
    return torch.einsum("bhtgl,blhd->bthgd", p, V.double()).reshape(B, T, Hq, D)


def accuracy_table(K, V, q, P=128, C=32, alpha=255.0, sweep=True):
    """vNMSE of the attention output (the metric of the pages' Table 3,
    [Review], Mechanism 3) for each codec, against attention over the BF16
    K and V: the linear INT8 / INT4 baselines (Eq. 4), the full Lynx code,
    and its Anchor alone at every bit split.  The codecs run through the
    library's kernels; only this evaluation's attention is plain float64.
    With `sweep`, the full code and the 4-bit Anchor over alpha x C x page.
    Bytes per element count the codes and their metadata."""
    import torch

    from split_stream_kv_gb300 import lynx
    L = K.shape[1]
    ref = _attention_f64(q, K, V)
    den = float((ref * ref).sum())

    def vn(Kh, Vh):
        o = _attention_f64(q, Kh, Vh)
        return float(((o - ref) ** 2).sum()) / den

    table = {}
    for bits in (8, 4):
        Kh = lynx.lynx_int_decode(*lynx.lynx_int_encode(K, bits), bits)
        Vh = lynx.lynx_int_decode(*lynx.lynx_int_encode(V, bits), bits)
        table[f"int{bits}"] = {"vnmse": vn(Kh, Vh), "bytes_per_elem": bits / 8 + 8 / 128}

    def lynx_rows(P_, C_, a_, splits):
        ks = lynx.lynx_encode(K, P_, C_, a_)
        vs = lynx.lynx_encode(V, P_, C_, a_)
        meta_b = 8 / P_ + 8 / C_
        out = {"full": {"vnmse": vn(lynx.lynx_decode_full(*ks, L, P_, C_, a_),
                                    lynx.lynx_decode_full(*vs, L, P_, C_, a_)),
                        "bytes_per_elem": 1 + meta_b}}
        for k in splits:
            kk, _ = lynx.lynx_split_bits(ks[0], ks[1], k)
            vk, _ = lynx.lynx_split_bits(vs[0], vs[1], k)
            out[k] = {"vnmse": vn(lynx.lynx_decode_anchor_bits(kk, ks[2], L, P_, C_, a_, k),
                                  lynx.lynx_decode_anchor_bits(vk, vs[2], L, P_, C_, a_, k)),
                      "anchor_bytes_per_elem": k / 8 + meta_b,
                      "total_bytes_per_elem": 1 + meta_b}
        return out

    ka1 = lynx.lynx_a1_encode(K, P, 100.0)
    va1 = lynx.lynx_a1_encode(V, P, 100.0)
    a1_meta = 4 * (1 + P // 16) / P
    table["a1_full"] = {"vnmse": vn(lynx.lynx_a1_decode(*ka1, L, P, 100.0),
                                    lynx.lynx_a1_decode(*va1, L, P, 100.0)),
                        "bytes_per_elem": 1 + a1_meta}
    table["a1_anchor"] = {"vnmse": vn(lynx.lynx_a1_decode(ka1[0], None, ka1[2], L, P, 100.0),
                                      lynx.lynx_a1_decode(va1[0], None, va1[2], L, P, 100.0)),
                          "anchor_bytes_per_elem": 0.5 + a1_meta}
    del ka1, va1
    rows = lynx_rows(P, C, alpha, (3, 4, 5, 6))
    table["lynx_full"] = rows["full"]
    for k in (3, 4, 5, 6):
        table[f"lynx_anchor_{k}bit"] = rows[k]
    if sweep:
        sw = []
        for a_ in (100.0, 500.0, 2000.0):
            for C_ in (16, 32, 64):
                for P_ in SWEEP_PAGES:
                    r = lynx_rows(P_, C_, a_, (4,))
                    sw.append({"alpha": a_, "C": C_, "page": P_,
                               "full_vnmse": r["full"]["vnmse"],
                               "anchor4_vnmse": r[4]["vnmse"],
                               "anchor_bytes_per_elem": r[4]["anchor_bytes_per_elem"]})
        table["sweep"] = sw
    torch.cuda.synchronize()
    return table


# page sizes of the ablation sweep ([Review], Concrete Improvement
# Suggestions, item 4)
SWEEP_PAGES = (128, 256, 512)


def measure_variants(c, kv, anc, res, meta, dev, reps=5):
    """HBM throughput of the comparison-point kernels on a codec workload:
    INT8 / INT4 encode and decode, the 6+2 and 3+5 re-splits and the k-bit
    Anchor decode.  Algorithmic bytes: what each kernel must read and write."""
    import torch

    from split_stream_kv_gb300 import lynx
    n = kv.numel()
    peak = load_peaks()[0]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timed(fn):
        return median_ms(fn, dev, reps, flush, warm=2)

    out = {}

    def row(name, fn, nbytes):
        ms = timed(fn)
        gbps = nbytes / ms / 1e6
        out[name] = {"ms": round(ms, 4), "algorithmic_bytes": int(nbytes),
                     "achieved_GBps": round(gbps, 1),
                     "roofline_frac": round(gbps / peak, 4) if peak else None}

    meta_b = n * (8 / c["P"] + 8 / c["C"])
    for bits in (8, 4):
        codes, m = lynx.lynx_int_encode(kv, bits)
        dec = torch.empty_like(kv)
        row(f"int{bits}_encode", lambda: lynx.lynx_int_encode(kv, bits, codes, m),
            n * (2 + bits / 8 + 8 / 128))
        row(f"int{bits}_decode", lambda: lynx.lynx_int_decode(codes, m, bits, out=dec),
            n * (bits / 8 + 8 / 128 + 2))
        del codes, m, dec
    a1 = lynx.lynx_a1_encode(kv, c["P"], 100.0)
    dec = torch.empty_like(kv)
    a1_meta = n * 4 * (1 + c["P"] // 16) / c["P"]
    row("a1_encode", lambda: lynx.lynx_a1_encode(kv, c["P"], 100.0), n * 3 + a1_meta)
    row("a1_decode_full", lambda: lynx.lynx_a1_decode(*a1, c["L"], c["P"], 100.0, out=dec),
        n * 3 + a1_meta)
    del a1, dec
    for k in (6, 5, 3):
        ak, rk = lynx.lynx_split_bits(anc, res, k)
        row(f"split_{k}+{8 - k}", lambda: lynx.lynx_split_bits(anc, res, k, ak, rk), n * 2)
        dec = torch.empty_like(kv)
        row(f"decode_anchor_{k}bit",
            lambda: lynx.lynx_decode_anchor_bits(ak, meta, c["L"], c["P"], c["C"], ALPHA, k,
                                                 out=dec),
            n * (k / 8 + 2) + meta_b)
        del ak, rk, dec
    del flush
    return out


def measure_split(c, kv, kv_h, dev_streams, host_streams, out, dev, reps=3,
                  pages_per_group=256):
    """The split-stream timeline on a codec workload, one GPU as either end
    of the link (pinned host memory standing in for it): the receiver's time
    until every Anchor group is on the device and decoded (when drafting can
    start) and until every group is upgraded to the full decode, against the
    time the BF16 tensor alone takes over the same link; and the sender's
    times for encode + copy-out.  Medians over `reps`, each from an event on
    the copy stream recorded before the first operation."""
    import torch

    from split_stream_kv_gb300 import lynx
    copy_s = torch.cuda.Stream(dev)
    hi = torch.cuda.Stream(dev, priority=-1)
    lo = torch.cuda.Stream(dev, priority=0)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def timed(fn, n_marks):
        res = []
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            e0 = ev()
            marks = [ev() for _ in range(n_marks)]
            e0.record(copy_s)
            fn(marks)
            torch.cuda.synchronize(dev)
            res.append([e0.elapsed_time(m) for m in marks])
        return [statistics.median(r[i] for r in res) for i in range(n_marks)]

    def bf16_in(m):
        with torch.cuda.stream(copy_s):
            kv.copy_(kv_h, non_blocking=True)
            m[0].record(copy_s)

    def bf16_out(m):
        with torch.cuda.stream(copy_s):
            kv_h.copy_(kv, non_blocking=True)
            m[0].record(copy_s)

    def receive(m, with_out):
        lynx.lynx_split_receive(host_streams, dev_streams, c["L"], c["P"], c["C"], ALPHA,
                                pages_per_group, out=out if with_out else None,
                                copy_stream=copy_s, hi_stream=hi, lo_stream=lo,
                                anchor_ready=m[0], full_ready=m[1])

    def send(m):
        lynx.lynx_split_send(kv, c["P"], c["C"], ALPHA, dev_streams, host_streams,
                             pages_per_group, hi_stream=hi, copy_stream=copy_s,
                             anchor_sent=m[0], all_sent=m[1])

    t_in, = timed(bf16_in, 1)
    t_out, = timed(bf16_out, 1)
    r_anchor, r_full = timed(lambda m: receive(m, True), 2)
    c_anchor, c_all = timed(lambda m: receive(m, False), 2)
    s_anchor, s_all = timed(send, 2)
    a_bytes = sum(t.nbytes for t in (host_streams[0], host_streams[2]))
    all_bytes = a_bytes + host_streams[1].nbytes
    return {
        "workload": codec_desc(c["name"], c),
        "pages_per_group": pages_per_group,
        "bf16_bytes": kv_h.nbytes, "anchor_phase_bytes": a_bytes, "all_bytes": all_bytes,
        "bf16_h2d_ms": round(t_in, 4), "bf16_d2h_ms": round(t_out, 4),
        "receive_anchor_ready_ms": round(r_anchor, 4),
        "receive_full_ready_ms": round(r_full, 4),
        "receive_copies_anchor_ms": round(c_anchor, 4), "receive_copies_all_ms": round(c_all, 4),
        "send_anchor_sent_ms": round(s_anchor, 4), "send_all_sent_ms": round(s_all, 4),
        "time_to_anchor_speedup_vs_bf16": round(t_in / r_anchor, 3),
        "link_h2d_GBps": round(kv_h.nbytes / t_in / 1e6, 1),
        "what": "one GPU as either end of the link: pinned host memory in between; receiver "
                "times to every Anchor decoded and to every group upgraded in place, sender "
                "times for encode + copy-out, against the BF16 tensor over the same link",
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["lynx", "reference"], default="lynx")
    ap.add_argument("--no-cpu", action="store_true", help="skip the cpu_baseline leg")
    ap.add_argument("--rows", default=",".join(ROWS), help="comma-separated subset of rows")
    ap.add_argument("--small", action="store_true", help="small workloads for profiling")
    ap.add_argument("--codec", default=HEADLINE, choices=sorted(CODEC_CONFIGS),
                    help="codec configuration of the step")
    args = ap.parse_args()
    args.rows = [r for r in args.rows.split(",") if r]
    unknown = [r for r in args.rows if r not in ROWS]
    if unknown:
        ap.error(f"unknown rows {unknown}")
    CODEC.clear()
    CODEC.update(CODEC_CONFIGS[args.codec], name=args.codec)
    if args.small:
        CODEC["B"] = min(CODEC["B"], 8)
        ATTN["batch"] = 2

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args, world)

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    r = run_lynx(args, rank, world, dev)

    if rank == 0:
        be = bf16_equiv_bytes()
        alg = algorithmic_bytes()
        peak, peak_kind = load_peaks()
        run_rows = list(r["row_ms"].keys())
        step_ms = r["ms_total"] / args.steps
        step_bytes = sum(be[n] for n in run_rows)
        value = whole_job_gbps(step_bytes, world, step_ms / 1e3)
        rows = {}
        for name in run_rows:
            ms = r["row_ms"][name]
            ach = alg[name] / (ms / 1e3) / 1e9
            d = {"ms": round(ms, 4), "bf16_equiv_GBps": round(be[name] / (ms / 1e3) / 1e9, 1),
                 "algorithmic_bytes": int(alg[name]), "achieved_GBps": round(ach, 1),
                 "roofline_frac": round(ach / peak, 4),
                 "dram_traffic_bytes": recorded_traffic(name, units_per_launch(name))}
            if name.startswith("attn"):
                T = ATTN["T_draft"] if name == "attn_draft" else ATTN["T_verify"]
                d["tokens_per_s"] = round(ATTN["batch"] * T / (ms / 1e3), 1)
                d["context_tokens_per_s"] = round(ATTN["batch"] * ATTN["L"] / (ms / 1e3), 1)
            rows[name] = d
        dom = max(run_rows, key=lambda n: r["row_ms"][n])
        ach = alg[dom] / (r["row_ms"][dom] / 1e3) / 1e9
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(step_ms, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic",
            "config": workload_config(),
            "rows": rows,
            "anchor_attention_tokens_per_s": rows.get("attn_draft", {}).get("tokens_per_s"),
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(ach, 1),
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": round(ach / peak, 4),
                         "traffic": recorded_traffic(dom, units_per_launch(dom))},
            "e2e": None if r["e2e_s"] is None else {
                "value": round(whole_job_gbps(step_bytes, world, r["e2e_s"]), 2), "unit": "GB/s",
                "steps": args.steps,
                "h2d_bytes_per_step": int(r["h2d"]), "d2h_bytes_per_step": int(r["d2h"])},
            "gpu_launches": r["launches"],
            "clocks": r["clocks"],
        }
        for key in ("parity", "configs", "extras"):
            if r.get(key):
                line[key] = r[key]
        if args.small:
            line["config"]["workload"] = "SMALL profiling case: " + line["config"]["workload"]
            line["config"]["small"] = {"codec_B": CODEC["B"], "attn_batch": ATTN["batch"]}
        if world == 1 and not args.no_cpu and not args.small:
            sample = CpuSample()
            v, cores, desc, _ = cpu_sample_run(target_s=12.0, sample=sample)
            v1, _, desc1, _ = cpu_sample_run(target_s=8.0, threads=1, sample=sample)
            line["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": cores,
                                    "kind": "oracle", "sample": desc,
                                    "single_thread": {"value": round(v1, 4), "unit": "GB/s",
                                                      "cores": 1, "sample": desc1}}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


# one reference step: this many passes over the fixed CPU sample
REFERENCE_PASSES = 24


def run_reference(args, world):
    """The reference arm: the CPU oracle on the host cores.  One step is a
    fixed sample of the same rows (REFERENCE_PASSES passes over the CPU
    sample), timed as it runs; the value is the sample's BF16-equivalent
    bytes over the measured time, reweighted to the step's byte mix."""
    sample = CpuSample()
    threads = os.cpu_count() or 1
    for _ in range(args.warmup):
        sample.run(threads)
    totals = [0.0, 0, 0.0, 0]
    step_s = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        for _ in range(REFERENCE_PASSES):
            for i, x in enumerate(sample.run(threads)):
                totals[i] += x
        step_s.append(time.perf_counter() - t0)
    value = step_rate(*totals)
    desc = (f"{REFERENCE_PASSES} x [{sample.desc()}] per step on {threads} threads; codec and "
            "attention rates reweighted to the step's byte mix")
    cfg = workload_config()
    cfg["reference_step"] = ("one step = the fixed CPU sample below (not the full workload); "
                             "ms_per_step is its measured wall time")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * sum(step_s) / len(step_s), 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
