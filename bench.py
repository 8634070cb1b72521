"""Benchmark of the split-stream KV hot path on GB300.

One step = every row of the path on synthetic data resident in HBM:
  encode        Llama-3-8B-shaped KV: 32 layers x (K, V) = B 64, L 16384,
                8 KV heads, D 128, page 128, C 32, alpha 255 (2 GiB BF16)
  decode_anchor the same streams -> BF16 KV
  decode_full   the same streams -> BF16 KV
  attn_draft    8 sequences x 32768 tokens, 32 query heads / 8 KV heads,
                T = 1 over the Anchor codes (+ split combine)
  attn_verify   the same KV, T = 8 over Anchor + Residual (+ split combine)
Metric: BF16-equivalent KV GB/s over the whole step (2 bytes per KV element
each row touches), with per-row times, roofline fractions of the measured HBM
bandwidth, and decode-attention tokens/s.

Flags: --gpus N (one replica per rank under torchrun; weak scaling),
--steps K, --warmup W, --impl {lynx,reference}.  --impl reference times the
CPU oracle (the only reference this path has) on a bounded sample.
Profiling aids: --rows a,b selects rows; --small shrinks both workloads (codec
B = 8, attention batch 2; still larger than L2) and skips the e2e and CPU legs.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV codec GB/s (BF16-equivalent) and anchor-attention tokens/s; % of HBM roofline"
ALPHA = 255.0
CODEC = dict(B=64, L=16384, H=8, D=128, P=128, C=32)
ATTN = dict(batch=8, L=32768, H_kv=8, H_q=32, D=128, P=128, C=32, T_draft=1, T_verify=8)


def meta_bytes_per_elem(P, C):
    return 8.0 / P + 8.0 / C


def codec_elems():
    return CODEC["B"] * CODEC["L"] * CODEC["H"] * CODEC["D"]


def attn_kv_elems():
    a = ATTN
    return 2 * a["batch"] * a["L"] * a["H_kv"] * a["D"]   # K and V


def algorithmic_bytes():
    """Bytes each row must move at minimum (per launch)."""
    n = codec_elems()
    m = meta_bytes_per_elem(CODEC["P"], CODEC["C"])
    na = attn_kv_elems()
    ma = meta_bytes_per_elem(ATTN["P"], ATTN["C"])
    return {
        "encode": n * (2 + 0.5 + 0.5 + m),
        "decode_anchor": n * (0.5 + m + 2),
        "decode_full": n * (0.5 + 0.5 + m + 2),
        "attn_draft": na * (0.5 + ma),
        "attn_verify": na * (1.0 + ma),
    }


def bf16_equiv_bytes():
    n = codec_elems()
    na = attn_kv_elems()
    return {"encode": 2 * n, "decode_anchor": 2 * n, "decode_full": 2 * n,
            "attn_draft": 2 * na, "attn_verify": 2 * na}


ROWS = ["encode", "decode_anchor", "decode_full", "attn_draft", "attn_verify"]


# Sources that define each row's kernel; the recorded DRAM traffic of a
# kernel is only reported while these files are unchanged.
ROW_SOURCES = {
    "encode": ["encode.cu", "common.cuh", "internal.h"],
    "decode_anchor": ["decode.cu", "common.cuh", "internal.h"],
    "decode_full": ["decode.cu", "common.cuh", "internal.h"],
    "attn_draft": ["attn.cu", "common.cuh", "internal.h"],
    "attn_verify": ["attn.cu", "common.cuh", "internal.h"],
}


def sources_hash(row):
    import hashlib
    h = hashlib.sha256()
    for name in ROW_SOURCES[row]:
        with open(os.path.join(ROOT, "split_stream_kv_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(row, units_per_launch):
    """DRAM bytes per launch of the row's kernel, scaled from the ncu capture
    recorded in profiles/traffic.md, or None if there is none for the current
    sources of the kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            cells = [c.strip() for c in line.strip().strip("|").split("|")]
            if len(cells) < 5 or cells[0] != row:
                continue
            try:
                sha, units, nbytes = cells[1], float(cells[2]), float(cells[3])
            except ValueError:
                continue
            if sha != sources_hash(row):
                return None
            return int(round(nbytes / units * units_per_launch))
    return None


def units_per_launch(row):
    """Elements (KV elements read or written) one launch of the row handles."""
    return codec_elems() if row in ("encode", "decode_anchor", "decode_full") else attn_kv_elems()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def workload_config():
    return {
        "workload": ("llama3-8b-shaped KV codec (B=64 = 32 layers x K,V; L=16384; H_kv=8; "
                     "D=128; page=128; C=32; alpha=255) + packed-KV decode attention "
                     "(8 seqs x 32768 tokens; H_q=32 over H_kv=8; draft T=1 anchor, "
                     "verify T=8 full)"),
        "l2": "inputs larger than L2 (2 GiB BF16 codec input, 0.69 GiB packed attention KV)",
        "parallelism": "replicas",
    }


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

def cpu_sample_run(target_s: float = 12.0, threads: int | None = None):
    """Time the oracle on a bounded sample of the step, repeated until about
    target_s seconds of work: page blocks of the codec workload (encode and
    both decodes of 2 x 4096 tokens x 8 heads) and attention of one
    (sequence, KV head) pair over 4096 tokens (both decoders of its pages,
    then the float64 softmax for the 4 draft rows and 32 verify rows).  The
    codec and attention rates are reweighted to the step's byte mix.  Returns
    (GB/s BF16-equivalent, threads, description, seconds)."""
    import numpy as np
    import torch

    import oracle
    from split_stream_kv_gb300 import synth

    threads = threads or (os.cpu_count() or 1)
    P, C = CODEC["P"], CODEC["C"]
    Lc = 4096
    kv = synth.kv_cache(2, Lc, CODEC["H"], 128, seed=11, device="cpu")
    bits = kv.view(torch.int16).numpy().view(np.uint16)
    La = 4096
    kva = synth.kv_cache(2, La, 1, 128, seed=5, device="cpu")
    ab = kva.view(torch.int16).numpy().view(np.uint16)
    ea, er, em = oracle.encode(ab, ATTN["P"], ATTN["C"], ALPHA, threads=threads)
    q = np.random.default_rng(0).standard_normal((ATTN["T_verify"] * 4, 128)).astype(np.float32)

    t_codec = t_attn = 0.0
    codec_bytes = attn_bytes = 0
    reps = 0
    while t_codec + t_attn < target_s or reps == 0:
        t0 = time.perf_counter()
        oa, orr, om = oracle.encode(bits, P, C, ALPHA, threads=threads)
        oracle.decode(oa, None, om, Lc, P, C, ALPHA, threads=threads)
        oracle.decode(oa, orr, om, Lc, P, C, ALPHA, threads=threads)
        t_codec += time.perf_counter() - t0
        codec_bytes += 3 * 2 * bits.size
        t0 = time.perf_counter()
        for full, rows in ((False, 4), (True, 4 * ATTN["T_verify"])):
            x = oracle.decode(ea, er if full else None, em, La, ATTN["P"], ATTN["C"], ALPHA,
                              threads=threads)
            xb = oracle.bf16_bits_to_f32(oracle.f32_to_bf16_bits(x)).reshape(x.shape)
            K, V = xb[0, :, 0], xb[1, :, 0]
            for r in range(rows):
                oracle.attention_row(q[r], K, V)
            attn_bytes += 2 * 2 * La * 128
        t_attn += time.perf_counter() - t0
        reps += 1
    be = bf16_equiv_bytes()
    w_codec = be["encode"] + be["decode_anchor"] + be["decode_full"]
    w_attn = be["attn_draft"] + be["attn_verify"]
    t_step = w_codec / (codec_bytes / t_codec) + w_attn / (attn_bytes / t_attn)
    value = (w_codec + w_attn) / t_step / 1e9
    desc = (f"{reps} x [{2 * (Lc // P) * CODEC['H']} page blocks (2 x {Lc} tokens x "
            f"{CODEC['H']} heads) encoded and decoded both ways + draft (4 rows) and verify "
            f"(32 rows) attention over one {La}-token (sequence, KV head) pair incl. its "
            f"decode]; {t_codec + t_attn:.1f} s on {threads} threads; codec and attention "
            f"rates reweighted to the step's byte mix")
    return value, threads, desc, t_codec + t_attn


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


def run_lynx(args, rank, world, dev):
    import torch

    from split_stream_kv_gb300 import lynx, synth

    torch.cuda.set_device(dev)
    c = CODEC
    a = ATTN
    kv = synth.kv_cache(c["B"], c["L"], c["H"], c["D"], seed=11 + rank, device=dev)
    anc, res, meta = lynx.lynx_encode(kv, c["P"], c["C"], ALPHA)
    dec_a = torch.empty_like(kv)
    dec_f = torch.empty_like(kv)
    kva = synth.kv_cache(2 * a["batch"], a["L"], a["H_kv"], a["D"], seed=5 + rank, device=dev)
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
    ws = torch.empty(ws_n, dtype=torch.uint8, device=dev)
    ks_anchor = (ks[0], None, ks[2])
    vs_anchor = (vs[0], None, vs[2])

    def row(name):
        if name == "encode":
            lynx.lynx_encode(kv, c["P"], c["C"], ALPHA, anc, res, meta)
        elif name == "decode_anchor":
            lynx.lynx_decode_anchor(anc, meta, c["L"], c["P"], c["C"], ALPHA, out=dec_a)
        elif name == "decode_full":
            lynx.lynx_decode_full(anc, res, meta, c["L"], c["P"], c["C"], ALPHA, out=dec_f)
        elif name == "attn_draft":
            lynx.lynx_attn_decode(q1, ks_anchor, vs_anchor, a["L"], a["P"], a["C"], ALPHA,
                                  lynx.LYNX_ANCHOR, out=out1, workspace=ws)
        else:
            lynx.lynx_attn_decode(q8, ks, vs, a["L"], a["P"], a["C"], ALPHA, lynx.LYNX_FULL,
                                  out=out8, workspace=ws)

    launches_per_step = {"encode": 1, "decode_anchor": 1, "decode_full": 1, "attn_draft": 2,
                         "attn_verify": 2}
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
    launches = sum(launches_per_step[r] for r in rows_run) * args.steps
    if args.small or rows_run != ROWS:
        ms_total, = max_over_ranks([ms_total], world, dev)
        return dict(ms_total=ms_total, row_ms=row_ms, e2e_s=None, h2d=0, d2h=0, clocks=clk,
                    launches=launches)

    # ---- end to end: pinned host buffers in, results out, every step
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
    nsl = 8 if c["B"] % 8 == 0 else 1
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

    e2e_steps = max(1, min(args.steps, 5))
    e2e_step()
    torch.cuda.synchronize(dev)
    barrier()
    w0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier()
    e2e_s = (time.perf_counter() - w0) / e2e_steps

    ms_total, e2e_s = max_over_ranks([ms_total, e2e_s], world, dev)
    extras = measure_extras(ks, vs, q8, ws, dev) if rank == 0 else None
    if extras is not None:
        extras["split_stream"] = measure_split(kv, kv_h, (anc, res, meta),
                                               (anc_h, res_h, meta_h), dec_a, dev)
        extras["variants"] = measure_variants(kv, anc, res, meta, dev)
        kva = synth.kv_cache(4, a["L"], a["H_kv"], a["D"], seed=5 + rank, device=dev)
        qa = synth.queries(2, a["T_verify"], a["H_q"], a["D"], seed=8, device=dev)
        extras["accuracy"] = accuracy_table(kva[0::2].contiguous(), kva[1::2].contiguous(), qa,
                                            a["P"], a["C"], ALPHA)
        extras["accuracy"]["what"] = (
            "vNMSE of attention outputs (2 sequences x 32768 tokens x 8 KV heads, 8 query "
            "tokens x 32 heads) against attention over the BF16 KV; codecs on the GPU")
        del kva
    assert lynx.lynx_wait_timeouts() == 0
    return dict(ms_total=ms_total, row_ms=row_ms, e2e_s=e2e_s, h2d=h2d, d2h=d2h, clocks=clk,
                launches=launches, extras=extras)


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
    verify_bytes = algorithmic_bytes()["attn_verify"]
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
                for P_ in (128, 256):
                    r = lynx_rows(P_, C_, a_, (4,))
                    sw.append({"alpha": a_, "C": C_, "page": P_,
                               "full_vnmse": r["full"]["vnmse"],
                               "anchor4_vnmse": r[4]["vnmse"],
                               "anchor_bytes_per_elem": r[4]["anchor_bytes_per_elem"]})
        table["sweep"] = sw
    torch.cuda.synchronize()
    return table


def measure_variants(kv, anc, res, meta, dev, reps=5):
    """HBM throughput of the comparison-point kernels on the codec workload:
    INT8 / INT4 encode and decode, the 6+2 and 3+5 re-splits and the k-bit
    Anchor decode.  Algorithmic bytes: what each kernel must read and write."""
    import statistics

    import torch

    from split_stream_kv_gb300 import lynx
    c = CODEC
    n = kv.numel()
    peak = load_peaks()[0]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        ts = []
        for i in range(reps + 2):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if i >= 2:
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

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


def measure_split(kv, kv_h, dev_streams, host_streams, out, dev, reps=3, pages_per_group=256):
    """The split-stream timeline on the codec workload, one GPU as either end
    of the link (pinned host memory standing in for it): the receiver's time
    until every Anchor group is on the device and decoded (when drafting can
    start) and until every group is upgraded to the full decode, against the
    time the BF16 tensor alone takes over the same link; and the sender's
    times for encode + copy-out.  Medians over `reps`, each from an event on
    the copy stream recorded before the first operation."""
    import statistics

    import torch

    from split_stream_kv_gb300 import lynx
    c = CODEC
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
    args = ap.parse_args()
    args.rows = [r for r in args.rows.split(",") if r]
    unknown = [r for r in args.rows if r not in ROWS]
    if unknown:
        ap.error(f"unknown rows {unknown}")
    if args.small:
        CODEC["B"] = 8
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
                "h2d_bytes_per_step": int(r["h2d"]), "d2h_bytes_per_step": int(r["d2h"])},
            "gpu_launches": r["launches"],
            "clocks": r["clocks"],
        }
        if r.get("extras"):
            line["extras"] = r["extras"]
        if args.small:
            line["config"]["workload"] = "SMALL profiling case: " + line["config"]["workload"]
            line["config"]["small"] = {"codec_B": CODEC["B"], "attn_batch": ATTN["batch"]}
        if world == 1 and not args.no_cpu and not args.small:
            v, cores, desc, _ = cpu_sample_run()
            line["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": cores,
                                    "kind": "oracle", "sample": desc}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_reference(args, world):
    """The reference arm: the CPU oracle on the host cores, each step a
    bounded sample of the same workload."""
    import oracle
    oracle.build()
    for _ in range(args.warmup):
        cpu_sample_run(target_s=1.0)
    vals, t_all = [], 0.0
    desc, cores = "", 0
    for _ in range(args.steps):
        v, cores, desc, t = cpu_sample_run(target_s=10.0)
        vals.append(v)
        t_all += t
    value = sum(vals) / len(vals)
    step_bytes = sum(bf16_equiv_bytes().values())
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_bytes / (value * 1e9) * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": workload_config(),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
