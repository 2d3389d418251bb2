"""Benchmark: one paged decode step (kv_append of each sequence's new token, then paged
GQA decode attention) on the Llama-3-8B layer shape, through libpkv's C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is K/V-cache bytes read per step divided by the
device time of a step, summed over ranks (replicas: every rank runs its own copy of the
workload, nothing is exchanged).  Where sequences share prefix blocks, each physical block
counts once (the bytes that must cross HBM); the logical bytes are given as `effective`.
Each timed step is bracketed by CUDA events on the launch stream; the L2 cache is flushed
between steps (outside the events) by reading a buffer twice its size (a read, so that no
write-back of the flush lands in the next step).  `e2e` repeats the measurement through the
Python/C-ABI calls with pinned host inputs copied in and the output copied back every step;
`steady` repeats the step thousands of times with clock samples under load.  The default
run also times every other workload (`other_configs`: ragged batch, Llama-3-70B long
context, Qwen2.5-7B prefix sharing with bf16 and FP8 pools and with copy-on-write, the
32-layer step, prefill and chunked prefill), each with its value, roofline fraction and
traffic ratio.  `--impl reference` times the fp64 CPU oracle on a bounded sample of the
same workload (one sequence per step).
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "decode-attn KV GB/s (% of HBM peak) and query-tokens/s, Llama-3-8B layer shape"
DEFAULT_WORKLOAD = "llama3_8b"
FALLBACK_HBM_GBS = 6800.0
DECODE_SOURCES = ("decode_kernels.cuh", "paged_decode.cu", "pkv_device.cuh", "tc_device.cuh")


# ------------------------------------------------------------------ helpers
def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def _hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def code_hash(names) -> str:
    """sha256 (16 hex digits) of the named csrc files' code: // comments, trailing blanks and
    empty lines are dropped, so an edit to comments alone keeps a profile's counters valid."""
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "paged_kv_cache_159_gb300", "csrc", name)) as f:
            for line in f:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def decode_source_hash() -> str:
    return code_hash(DECODE_SOURCES)


def _profiled_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken on the
    current decode sources (else None)."""
    path = os.path.join(ROOT, "profiles", "decode_%s.md" % workload)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    s = re.search(r"decode_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != decode_source_hash():
        return None
    return int(m.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms in the background."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def reduce_max_over_ranks(values, device):
    """Elementwise max of per-rank timings (the slowest rank sets the step time)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def aggregate_value(world, kv_bytes_per_step, steps, slowest_total_s):
    """Whole-job GB/s: every rank's bytes over the slowest rank's time (weak scaling)."""
    return world * kv_bytes_per_step * steps / slowest_total_s / 1e9


# ------------------------------------------------------------------ our arm
def _unique_kv_positions(tables, seq_lens, num_blocks):
    """Positions of K/V read when every physical block is read once: for each distinct block
    id, the most positions any sequence reads from it.  A block shared by many tables (a
    common prefix) counts once, as the pages store it once."""
    most = np.zeros(num_blocks, np.int64)
    for b, L in enumerate(seq_lens):
        nb = -(-int(L) // 16)
        np.maximum.at(most, tables[b, :nb], np.minimum(16, int(L) - 16 * np.arange(nb)))
    return int(most.sum())


def _copy_probe(pkv, torch, dev, stream):
    """The library's streaming copy over 2 x 1 GiB, best of 10: the same-process bandwidth
    denominator reported beside the measured peak."""
    src = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    dst = torch.empty_like(src)
    for _ in range(3):
        pkv.probe_copy(dst, src, stream=stream)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    probe = []
    with torch.cuda.stream(stream):
        for _ in range(10):
            ev[0].record(stream)
            pkv.probe_copy(dst, src, stream=stream)
            ev[1].record(stream)
            ev[1].synchronize()
            probe.append(ev[0].elapsed_time(ev[1]) * 1e-3)
    copy_gbs = 2 * src.numel() / min(probe) / 1e9
    del src, dst
    return copy_gbs


def run_decode(args, name, world, rank, local_rank, K, W, full=True):
    """One decode workload: K timed steps after W warm-up steps.  full: also the end-to-end
    leg from host memory, the steady repeat with clock samples and the oracle on the host."""
    import torch
    import paged_kv_cache_159_gb300 as pkv

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = workloads.WORKLOADS[name]
    nl = w.layers
    if nl > 1 and w.kv_dtype == "fp8":
        raise SystemExit("layered workloads are bf16")
    d = workloads.draw(w, dev)
    B, Hq, D = d.q.shape[-3:]
    Hkv = w.num_kv_heads
    elem = 1 if w.kv_dtype == "fp8" else 2

    # pool, block tables and slots from the library's host allocator
    k_scale = v_scale = 1.0
    kc, vc = d.key_cache, d.value_cache
    if w.kv_dtype == "fp8":
        k_scale = float(np.float32(kc.float().abs().max().item()) / np.float32(448.0))
        v_scale = float(np.float32(vc.float().abs().max().item()) / np.float32(448.0))
    pool = pkv.Pool(d.num_blocks, Hkv, D, pkv.KV_FP8E4M3 if w.kv_dtype == "fp8" else pkv.KV_BF16,
                    k_scale, v_scale, d.free_order, num_layers=nl)
    pool.attach_device(local_rank)
    prefix = pool.alloc(w.prefix_blocks) if w.prefix_blocks else None
    tables = pool.build_block_tables(d.seq_lens, d.max_blocks, prefix)
    cow_pairs = np.zeros((0, 2), np.int32)
    if w.append and w.prefix_blocks:
        # sequences whose newest position lies in a shared block diverge: copy-on-write
        # bookkeeping once on the host; the block copies run in every timed step (each step
        # is the step in which those sequences diverge)
        tables, cow_pairs = pool.cow_prepare(tables, d.seq_lens)
    slots = pkv.slot_mapping(tables, d.seq_lens)
    if w.kv_dtype == "fp8":                      # encode the history through kv_append
        alls = torch.from_numpy(pkv.slot_mapping_all(tables, d.seq_lens)).to(dev)
        k8 = torch.zeros(kc.shape, dtype=torch.uint8, device=dev)
        v8 = torch.zeros_like(k8)
        for i in range(0, alls.numel(), 1 << 16):
            s = alls[i:i + (1 << 16)]
            pkv.kv_append(pool, kc[s // 16, :, s % 16, :].contiguous(),
                          vc[s // 16, :, s % 16, :].contiguous(), s, k8, v8)
        kc, vc = k8, v8
        del d.key_cache, d.value_cache
    bt = torch.from_numpy(tables).to(dev)
    sl = torch.from_numpy(d.seq_lens).to(dev)
    sm = torch.from_numpy(slots).to(dev)
    out = torch.empty_like(d.q)
    decode_opts = json.loads(args.opts) if args.opts else None
    ws_bytes = pkv.decode_workspace_bytes(pool, B, Hq, d.max_blocks, decode_opts)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    cow_src = torch.from_numpy(cow_pairs[:, 0].copy()).to(dev)
    cow_dst = torch.from_numpy(cow_pairs[:, 1].copy()).to(dev)
    launches_per_step = ((1 if w.append and args.separate_append else 0) + 1 + (1 if len(cow_pairs) else 0) +
                         (1 if (decode_opts or {}).get("shared_prefix_blocks", 0) else 0))
    # algorithmic bytes (no credit for tail-slot over-read; shared prefix blocks counted
    # once per reader here, i.e. logical bytes); every layer reads its own K/V, queries and
    # outputs, and all layers share one read of the tables
    kv_read = nl * int(d.seq_lens.astype(np.int64).sum()) * Hkv * D * elem * 2
    decode_bytes = kv_read + nl * 2 * B * Hq * D * 2 + B * d.max_blocks * 4 + B * 4
    new_rows = nl * 2 * B * Hkv * D * (2 + elem)              # read k/v_new, write the rows
    append_bytes = (new_rows + (B * 8 if args.separate_append else 0)) if w.append else 0
    cow_bytes = 2 * 2 * len(cow_pairs) * pool.layer_bytes() // d.num_blocks * nl   # K+V, read+write
    step_bytes = decode_bytes + append_bytes + cow_bytes
    # bytes of the timed decode launch: with decode_step it also reads k_new/v_new and writes
    # the new rows
    launch_bytes = decode_bytes + (new_rows if w.append and not args.separate_append else 0)

    # the step's device inputs; the end-to-end leg below passes views of one packed buffer
    dev_in = {"q": d.q, "k": d.k_new, "v": d.v_new, "bt": bt, "sl": sl, "sm": sm, "cs": cow_src, "cd": cow_dst}

    def cow_call(stream=None, t=dev_in):
        if len(cow_pairs):
            pkv.copy_blocks(pool, kc, vc, t["cs"], t["cd"], stream=stream)

    def append_call(stream=None, t=dev_in):
        if nl > 1:
            pkv.kv_append_layers(pool, t["k"], t["v"], t["sm"], kc, vc, stream=stream)
        else:
            pkv.kv_append(pool, t["k"], t["v"], t["sm"], kc, vc, stream=stream)

    def decode_call(fused: bool, stream=None, t=dev_in):
        if nl > 1:
            pkv.decode_step_layers(pool, t["q"], t["k"] if fused else None, t["v"] if fused else None,
                                   kc, vc, t["bt"], t["sl"], w.scale, out, ws, opts=decode_opts, stream=stream)
        elif fused:
            pkv.decode_step(pool, t["q"], t["k"], t["v"], kc, vc, t["bt"], t["sl"], w.scale, out, ws,
                            opts=decode_opts, stream=stream)
        else:
            pkv.paged_attention_decode(pool, t["q"], kc, vc, t["bt"], t["sl"], w.scale, out, ws, opts=decode_opts,
                                       stream=stream)

    # same-process bandwidth denominator: the library's copy probe over 2 x 1 GiB
    copy_gbs = None
    if full:
        copy_gbs = _copy_probe(pkv, torch, dev, stream)

    # L2 flush between steps: a read of a buffer twice the L2 size.  Reading leaves only clean
    # lines behind, so no write-back of the flush lands inside the next timed step.
    flush_buf = torch.ones(2 * torch.cuda.get_device_properties(dev).L2_cache_size // 4,
                           dtype=torch.int32, device=dev)
    flush_out = torch.empty((), dtype=torch.int64, device=dev)

    def flush_l2():
        torch.sum(flush_buf, dim=0, out=flush_out)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]

    def timed_step(i, starts=starts, mids=mids, ends=ends):
        flush_l2()                                # L2 flush (read), outside the timed interval
        starts[i].record(stream)
        cow_call(stream)
        if w.append and args.separate_append:
            append_call(stream)
        mids[i].record(stream)
        decode_call(w.append and not args.separate_append, stream)   # fused: one launch
        ends[i].record(stream)

    with torch.cuda.stream(stream):
        for i in range(W):
            timed_step(i % K)
    stream.synchronize()
    st, bits = pool.get_device_error(stream)
    if st != pkv.OK:
        raise RuntimeError("device error in warm-up: %d bits %#x" % (st, bits))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for i in range(K):
                timed_step(i)
        stream.synchronize()
        wall = time.perf_counter() - t0
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    step_s = [starts[i].elapsed_time(ends[i]) * 1e-3 for i in range(K)]
    dec_s = [mids[i].elapsed_time(ends[i]) * 1e-3 for i in range(K)]
    total = float(sum(step_s))
    dec_mean = float(sum(dec_s) / K)
    st, bits = pool.get_device_error(stream)
    if st != pkv.OK:
        raise RuntimeError("device error in the timed region: %d bits %#x" % (st, bits))

    # ---- the steady repeat of the same step: enough steps for clock samples under load
    steady = None
    if full and args.steady_steps > 0:
        S = args.steady_steps
        st_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(S)] for _ in range(3)]
        with ClockSampler(local_rank) as sclk:
            with torch.cuda.stream(stream):
                for i in range(S):
                    timed_step(i, *st_ev)
            stream.synchronize()
        st_step = sorted(st_ev[0][i].elapsed_time(st_ev[2][i]) * 1e-3 for i in range(S))
        st_dec = sorted(st_ev[1][i].elapsed_time(st_ev[2][i]) * 1e-3 for i in range(S))
        steady = {"steps": S, "ms_per_step_median": round(st_step[S // 2] * 1e3, 5),
                  "kernel_us_median": round(st_dec[S // 2] * 1e6, 2),
                  "clocks": sclk.summary()}
        st, bits = pool.get_device_error(stream)
        if st != pkv.OK:
            raise RuntimeError("device error in the steady repeat: %d bits %#x" % (st, bits))

    def e2e_leg():
        # ---- end to end through the API: pinned host inputs in, output back, every step
        host = {}
        pin = lambda t: t.detach().cpu().pin_memory()
        host["q"], host["k"], host["v"] = pin(d.q), pin(d.k_new), pin(d.v_new)
        host["sl"] = torch.from_numpy(d.seq_lens.copy()).pin_memory()
        host["out"] = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        tables_host = tables
        h2d = (host["q"].numel() * 2 + (host["k"].numel() * 2 * 2 if w.append else 0)
               + tables_host.nbytes + host["sl"].numel() * 4
               + (B * 8 if w.append and args.separate_append else 0) + cow_pairs.nbytes)
        d2h = host["out"].numel() * 2
        cow_src_h = torch.from_numpy(cow_pairs[:, 0].copy()).pin_memory()
        cow_dst_h = torch.from_numpy(cow_pairs[:, 1].copy()).pin_memory()
        e2e_steps = max(5, min(K, 200))
        bt_h = torch.from_numpy(tables_host).pin_memory()
        sm_h = torch.empty(B, dtype=torch.int64).pin_memory()
        ee = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        e2e_t = []
        # the one-call host-memory step (pkv_decode_step_host) where it covers the step: copies
        # in, the one-launch step and the copy out issued by one C call
        one_call = nl == 1 and not args.separate_append and not len(cow_pairs)
        if one_call:
            # the step's inputs laid out back to back in one pinned host buffer and one device
            # buffer (q, k_new, v_new, block_tables, seq_lens): one upload per step
            parts = [("q", host["q"])] + ([("k_new", host["k"]), ("v_new", host["v"])] if w.append else []) + \
                    [("block_tables", bt_h), ("seq_lens", host["sl"])]
            sizes = [t.numel() * t.element_size() for _, t in parts]
            hbuf = torch.empty(sum(sizes), dtype=torch.uint8).pin_memory()
            dbuf = torch.empty(sum(sizes), dtype=torch.uint8, device=dev)
            hstep, dstep, off = {"out": host["out"], "contiguous": True}, {"out": out}, 0
            for (name, t), n in zip(parts, sizes):
                hv = hbuf[off:off + n].view(t.dtype).view(t.shape)
                hv.copy_(t)
                hstep[name] = hv
                dstep[name] = dbuf[off:off + n].view(t.dtype).view(t.shape)
                off += n
            # the call prepared once for these buffers (as a serving loop would); each step is
            # still one C call that uploads the inputs, decodes and downloads the output
            prepared = pkv.DecodeStepHost(pool, hstep, dstep, kc, vc, w.scale, ws, opts=decode_opts,
                                          stream=torch.cuda.current_stream())
        else:
            # the other steps (copy-on-write, a separate append, several layers): the inputs are
            # packed the same way, one upload per step, and the library calls take views of the
            # device copy
            parts = [("q", host["q"])] + ([("k", host["k"]), ("v", host["v"])] if w.append else []) + \
                    [("bt", bt_h), ("sl", host["sl"])] + \
                    ([("cs", cow_src_h), ("cd", cow_dst_h)] if len(cow_pairs) else []) + \
                    ([("sm", sm_h)] if w.append and args.separate_append else [])
            spans = [(t.numel() * t.element_size() + 15) // 16 * 16 for _, t in parts]   # 16-byte aligned views
            hbuf = torch.empty(sum(spans), dtype=torch.uint8).pin_memory()
            dbuf = torch.empty(sum(spans), dtype=torch.uint8, device=dev)
            hview, dview, off = {}, dict(dev_in), 0
            for (name, t), n in zip(parts, spans):
                nb = t.numel() * t.element_size()
                hview[name] = hbuf[off:off + nb].view(t.dtype).view(t.shape)
                hview[name].copy_(t)
                dview[name] = dbuf[off:off + nb].view(t.dtype).view(t.shape)
                off += n
            h2d = int(hbuf.numel())                   # the packed buffer is what is uploaded
        ref_out = out.detach().cpu()                  # the timed steps' output
        for i in range(e2e_steps + 3):
            flush_l2()
            torch.cuda.synchronize()
            ee[0].record()
            if one_call:
                prepared.run()                                                 # one upload, one download
                ee[1].record()
                ee[1].synchronize()
                if i >= 3:
                    e2e_t.append(ee[0].elapsed_time(ee[1]) * 1e-3)
                continue
            if w.append and args.separate_append:
                slots_np = pkv.slot_mapping(tables_host, d.seq_lens)        # host allocator side
                hview["sm"][:] = torch.from_numpy(slots_np)
            dbuf.copy_(hbuf, non_blocking=True)                              # one upload
            if w.append:
                cow_call(t=dview)
                if args.separate_append:
                    append_call(t=dview)
                    decode_call(False, t=dview)
                else:
                    decode_call(True, t=dview)
            else:
                decode_call(False, t=dview)
            host["out"].copy_(out, non_blocking=True)
            ee[1].record()
            ee[1].synchronize()
            if i >= 3:
                e2e_t.append(ee[0].elapsed_time(ee[1]) * 1e-3)
        e2e_step = float(statistics.median(e2e_t))
        if not torch.equal(host["out"].view(torch.int16), ref_out.view(torch.int16)):
            raise RuntimeError("end-to-end decode output differs from the timed steps'")
        api = ("DecodeStepHost.run (one pkv_decode_step_host call)" if one_call
               else "one packed upload + library calls on views of it")
        serial = None
        if one_call:
            # The same steps as a serving loop pipelines them: step i+1's upload overlaps step
            # i's decode and step i-1's download (three streams, two sets of device buffers);
            # the decodes stay in order on one stream, and a set is refilled only once its
            # decode and download are done.  Every step still uploads its inputs and downloads
            # its output.  No L2 flush between pipelined steps: the inputs exceed L2.
            serial = (e2e_step, api)
            sets = []
            for _ in range(2):
                db = torch.empty_like(dbuf)
                views, off = {}, 0
                for (name, t), n in zip(parts, sizes):
                    views[name] = db[off:off + n].view(t.dtype).view(t.shape)
                    off += n
                sets.append({"buf": db, "v": views, "out": torch.empty_like(out), "ws": torch.zeros_like(ws),
                             "hout": torch.empty(out.shape, dtype=out.dtype).pin_memory()})
            s_up, s_run, s_down = (torch.cuda.Stream(device=dev) for _ in range(3))
            n = e2e_steps
            ev_in, ev_run, ev_down = ([torch.cuda.Event() for _ in range(n)] for _ in range(3))
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            for _ in range(2):                                  # the first pass warms up
                torch.cuda.synchronize()
                t0.record(s_up)
                for i in range(n):
                    st = sets[i & 1]
                    if i >= 2:
                        s_up.wait_event(ev_run[i - 2])          # the set's inputs are read
                    with torch.cuda.stream(s_up):
                        st["buf"].copy_(hbuf, non_blocking=True)
                    ev_in[i].record(s_up)
                    s_run.wait_event(ev_in[i])
                    if i >= 2:
                        s_run.wait_event(ev_down[i - 2])        # the set's output is downloaded
                    v = st["v"]
                    if w.append:
                        pkv.decode_step(pool, v["q"], v["k_new"], v["v_new"], kc, vc, v["block_tables"],
                                        v["seq_lens"], w.scale, st["out"], st["ws"], opts=decode_opts, stream=s_run)
                    else:
                        pkv.paged_attention_decode(pool, v["q"], kc, vc, v["block_tables"], v["seq_lens"], w.scale,
                                                   st["out"], st["ws"], opts=decode_opts, stream=s_run)
                    ev_run[i].record(s_run)
                    s_down.wait_event(ev_run[i])
                    with torch.cuda.stream(s_down):
                        st["hout"].copy_(st["out"], non_blocking=True)
                    ev_down[i].record(s_down)
                t1.record(s_down)
                t1.synchronize()
            e2e_step = t0.elapsed_time(t1) * 1e-3 / n
            for st in sets:
                if not torch.equal(st["hout"].view(torch.int16), ref_out.view(torch.int16)):
                    raise RuntimeError("pipelined end-to-end decode output differs from the timed steps'")
            api = ("torch uploads and downloads + pkv.%s, pipelined over three streams and two buffer sets"
                   % ("decode_step" if w.append else "paged_attention_decode"))
        return e2e_step, h2d, d2h, api, serial

    e2e_step = h2d = d2h = e2e_serial = None
    if full:
        e2e_step, h2d, d2h, e2e_api, e2e_serial = e2e_leg()

    # ---- reduce over ranks (max time), aggregate bytes over ranks
    if world > 1:
        total, dec_mean = reduce_max_over_ranks([total, dec_mean], dev)
        if e2e_step is not None:
            (e2e_step,) = reduce_max_over_ranks([e2e_step], dev)
    peak, peak_src = _hbm_peak()
    ms_per_step = total / K * 1e3
    # Shared prefix blocks are stored once and read by many tables: their bytes cross HBM
    # once, so the roofline counts unique K/V bytes (each physical block once); the logical
    # bytes (every table's view) are reported beside them as "effective".
    shared = w.prefix_blocks > 0
    kv_unique = (nl * _unique_kv_positions(tables, d.seq_lens, d.num_blocks) * Hkv * D * elem * 2
                 if shared else kv_read)
    launch_unique = launch_bytes - kv_read + kv_unique
    value = aggregate_value(world, kv_unique, K, total)
    achieved = launch_unique / dec_mean / 1e9
    traffic = _profiled_traffic(name)
    variant = (decode_opts or {}).get("variant", 0) or 3
    kernel = "%s (%s%s)" % ({1: "decode_simt_kernel", 2: "decode_mma_kernel", 3: "decode_tok_kernel"}[variant],
                            "decode_step" if w.append and not args.separate_append
                            else "paged_attention_decode", ", %d layers" % nl if nl > 1 else "")
    step = (("copy_blocks + " if len(cow_pairs) else "") +
            (("kv_append + paged_attention_decode" if args.separate_append else
              "decode_step (append at L-1 + paged decode, one launch)") if w.append
             else "paged_attention_decode") + (", all %d layers per launch" % nl if nl > 1 else ""))
    basis = ("unique K/V bytes (each shared prefix block once)" if shared else "K/V bytes")
    if not full:
        r = {"value": round(value, 1), "unit": "GB/s", "basis": basis, "step": step,
             "ms_per_step": round(ms_per_step, 5), "kernel_us": round(dec_mean * 1e6, 2),
             "frac": round(achieved / peak, 4), "achieved": round(achieved, 1),
             "bytes_per_launch": launch_unique,
             "traffic": traffic, "traffic_ratio": round(traffic / launch_unique, 3) if traffic else None,
             "kernel": kernel, "steps": K, "warmup": W, "gpu_launches": launches_per_step * K,
             "query_tokens_per_s": round(world * B * K / total, 1)}
        if shared:
            r["effective"] = round(aggregate_value(world, kv_read, K, total), 1)
            r["effective_basis"] = "logical K/V bytes (every table's blocks counted)"
            r["effective_frac"] = round(launch_bytes / dec_mean / 1e9 / peak, 4)
        return r
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8e4m3-kv/bf16-q" if w.kv_dtype == "fp8" else "bf16", "data": "synthetic",
        "config": {
            "workload": "%s: %sbatch %d, q heads %d / kv heads %d, head_dim %d, block 16, "
                        "seq_lens %s, kv %s" % (w.name, "%d layers, " % nl if nl > 1 else "", B, Hq, Hkv, D,
                                                 "all %d" % d.seq_lens[0] if w.lengths == "fixed"
                                                 else "%s (sum %d)" % (w.lengths, int(d.seq_lens.sum())),
                                                 w.kv_dtype),
            "copy_on_write_pairs": int(len(cow_pairs)),
            "step": step,
            "decode_opts": decode_opts,
            "l2": "flushed between steps (read of a 2x L2 buffer); inputs also exceed L2",
            "parallelism": "replicas",
            "timing": "CUDA events around each step on the launch stream; flush outside them",
        },
        "basis": basis,
        "pct_of_hbm_peak": round(100.0 * (kv_unique * K / total / 1e9) / peak, 2),
        "query_tokens_per_s": round(world * B * K / total, 1),
        "step_bytes": step_bytes,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": kernel, "bytes_per_launch": launch_unique,
                     "peak_source": peak_src + " hbm_gbs", "same_run_copy_gbs": round(copy_gbs, 1) if copy_gbs else None},
        "e2e": {"value": round(world * kv_unique / e2e_step / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e2e_step * 1e3, 4), "api": e2e_api,
                **({"l2": "not flushed between pipelined steps (the inputs exceed L2)",
                    "serial": {"value": round(world * kv_unique / e2e_serial[0] / 1e9, 1),
                               "ms_per_step": round(e2e_serial[0] * 1e3, 4), "api": e2e_serial[1],
                               "l2": "flushed before each step; its copies and decode in series"}}
                   if e2e_serial else {})},
        "gpu_launches": launches_per_step * K,
        "clocks": clk.summary(),
        "wall_s_timed_region": round(wall, 3),
    }
    if shared:
        res["effective"] = round(aggregate_value(world, kv_read, K, total), 1)
        res["effective_basis"] = "logical K/V bytes (every table's blocks counted)"
    if steady is not None:
        steady["value_at_median"] = round(world * kv_unique / (steady["ms_per_step_median"] * 1e-3) / 1e9, 1)
        res["steady"] = steady
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, sample_seqs=args.cpu_sample_seqs)
    return res


# ------------------------------------------------------------------ the oracle on host cores
def _oracle_case(w, nseq):
    """A bounded sample of the workload for the oracle: the first `nseq` sequences."""
    import torch
    import oracle
    L = workloads.draw_seq_lens(w)[:nseq]
    sub = workloads.Workload(**{**w.__dict__, "batch": nseq, "lengths": "list",
                                "len_list": tuple(int(x) for x in L), "pool": "exact",
                                "prefix_blocks": 0, "layers": 1})
    d = workloads.draw(sub, "cpu")
    a = oracle.BlockAllocator(d.num_blocks, d.free_order)
    tables = oracle.build_block_tables(a, d.seq_lens, d.max_blocks)
    kb, vb = workloads.bf16_bits(d.key_cache), workloads.bf16_bits(d.value_cache)
    return sub, d, tables, kb, vb


def cpu_baseline(w, sample_seqs=64, threads=None, reps=3):
    import oracle
    threads = threads or os.cpu_count() or 1
    sample_seqs = min(sample_seqs, w.batch)
    sub, d, tables, kb, vb = _oracle_case(w, sample_seqs)
    q = workloads.bf16_bits(d.q)
    kn, vn = workloads.bf16_bits(d.k_new), workloads.bf16_bits(d.v_new)
    slots = oracle.slot_mapping(tables, d.seq_lens)
    t = []
    for _ in range(reps):
        t0 = time.perf_counter()
        if w.append:
            oracle.kv_append(kn, vn, slots, kb, vb)
        st, _ = oracle.paged_decode(q, kb, vb, tables, d.seq_lens, w.scale, w.num_kv_heads,
                                    num_threads=threads)
        t.append(time.perf_counter() - t0)
    sec = min(t)
    kv_read = int(d.seq_lens.astype(np.int64).sum()) * w.num_kv_heads * w.head_dim * 2 * 2
    # the same decode on one core, over the first sequences of the sample (at most 8)
    n1 = min(8, sample_seqs)
    pairs = np.array([[b, h] for b in range(n1) for h in range(w.num_q_heads)], dtype=np.int32)
    t0 = time.perf_counter()
    oracle.paged_decode(q, kb, vb, tables, d.seq_lens, w.scale, w.num_kv_heads, pairs=pairs, num_threads=1)
    sec1 = time.perf_counter() - t0
    kv1 = int(d.seq_lens[:n1].astype(np.int64).sum()) * w.num_kv_heads * w.head_dim * 2 * 2
    return {"value": round(kv_read / sec / 1e9, 4), "unit": "GB/s", "cores": int(threads),
            "kind": "oracle",
            "sample": "%d of %d sequences (all %d query heads), kv_append + fp64 decode, best of %d: %.3f s"
                      % (sample_seqs, w.batch, w.num_q_heads, reps, sec),
            "query_tokens_per_s": round(sample_seqs / sec, 2),
            "value_1core": round(kv1 / sec1 / 1e9, 4),
            "sample_1core": "%d sequences, fp64 decode on one core: %.3f s" % (n1, sec1),
            "cpu": _cpu_model()}


def _cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (model name, or the Arm implementer and part)."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                k, v = k.strip(), v.strip()
                if k and v and k not in fields:
                    fields[k] = v
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        return "%s, CPU implementer %s, part %s" % (platform.machine(), fields.get("CPU implementer", "?"), fields["CPU part"])
    return platform.machine()


def run_reference(args):
    """The oracle as the reference arm: each step is one sequence of the workload (all its
    query heads, kv_append + decode) in fp64 on the host cores."""
    import oracle
    w = workloads.WORKLOADS[args.workload]
    threads = os.cpu_count() or 1
    nseq = min(w.batch, 8)
    sub, d, tables, kb, vb = _oracle_case(w, nseq)
    q = workloads.bf16_bits(d.q)
    kn, vn = workloads.bf16_bits(d.k_new), workloads.bf16_bits(d.v_new)
    slots = oracle.slot_mapping(tables, d.seq_lens)
    per_seq_bytes = [int(L) * w.num_kv_heads * w.head_dim * 2 * 2 for L in d.seq_lens]

    def one(i):
        b = i % nseq
        pairs = np.array([[b, h] for h in range(w.num_q_heads)], dtype=np.int32)
        if w.append:
            oracle.kv_append(kn[b:b + 1], vn[b:b + 1], slots[b:b + 1], kb, vb)
        st, _ = oracle.paged_decode(q, kb, vb, tables, d.seq_lens, w.scale, w.num_kv_heads,
                                    pairs=pairs, num_threads=threads)
        return per_seq_bytes[b]

    for i in range(args.warmup):
        one(i)
    nbytes = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        nbytes += one(i)
    total = time.perf_counter() - t0
    value = nbytes / total / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "parallelism": "host threads",
                   "sample": "one sequence per step (all query heads, kv_append + decode)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": "one of the first %d sequences per step, %d steps" % (nseq, args.steps)},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "query_tokens_per_s": round(args.steps / total, 3),
    }


# ------------------------------------------------------------------ prefill workloads
PREFILL_METRIC = "prefill attention TFLOP/s (causal, visible keys only), Llama-3-8B layer shape"


def _prefill_flops(d, Hq, D):
    """Algorithmic FLOPs: every packed row sees positions 0 .. its own, and each visible key
    costs 2*D for q.K and 2*D for p.V per query head."""
    vis = 0
    for b in range(len(d.seq_lens)):
        P, L = int(d.chunk_lens[b]), int(d.seq_lens[b])
        C = L - P
        vis += P * C + P * (P + 1) // 2
    return 4 * Hq * D * vis


def _tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured bf16_tflops (burst)"
    except Exception:
        return 1900.0, "fallback"


def _prefill_oracle_sample(w, nrows=48, threads=None):
    """The oracle on a bounded sample: the last nrows rows of the first sequence (the rows
    with the most visible keys), timed once.  Returns (TFLOP/s, seconds, rows)."""
    import oracle
    d = workloads.draw_prefill(w, "cpu")
    a = oracle.BlockAllocator(d.num_blocks, d.free_order)
    t = oracle.build_block_tables(a, d.seq_lens, d.max_blocks)
    kb, vb = workloads.bf16_bits(d.key_cache), workloads.bf16_bits(d.value_cache)
    P, L = int(d.chunk_lens[0]), int(d.seq_lens[0])
    nrows = min(nrows, P)
    pos = np.arange(L - nrows, L)
    rows = pos - (L - P)
    q = workloads.bf16_bits(d.q)[rows]
    threads = threads or os.cpu_count() or 1
    dt, ks, vs = oracle.BF16, 1.0, 1.0
    if w.kv_dtype == "fp8":
        # the E4M3 pool of the GPU run, for sequence 0's positions (encoded outside the timing)
        ks = float(np.float32(max(d.key_cache.float().abs().max().item(), d.k_chunk.float().abs().max().item()))
                   / np.float32(448.0))
        vs = float(np.float32(max(d.value_cache.float().abs().max().item(), d.v_chunk.float().abs().max().item()))
                   / np.float32(448.0))
        sl = oracle.all_slots(t[:1], d.seq_lens[:1])
        k8, v8 = np.zeros(kb.shape, np.uint8), np.zeros(vb.shape, np.uint8)
        assert oracle.kv_append(kb[sl // 16, :, sl % 16, :], vb[sl // 16, :, sl % 16, :], sl, k8, v8, 16,
                                oracle.FP8E4M3, ks, vs) == 0
        kb, vb, dt = k8, v8, oracle.FP8E4M3
    t0 = time.perf_counter()
    st, _ = oracle.paged_decode(q, kb, vb, np.repeat(t[:1], nrows, 0), (pos + 1).astype(np.int32), w.scale,
                                w.num_kv_heads, 16, dt, ks, vs, num_threads=threads)
    sec = time.perf_counter() - t0
    flops = 4 * w.num_q_heads * w.head_dim * int((pos + 1).sum())
    return flops / sec / 1e12, sec, nrows, threads


PREFILL_SOURCES = ("prefill.cu", "tc_device.cuh", "pkv_device.cuh")


def _prefill_traffic(workload: str):
    """DRAM bytes per prefill launch from the committed ncu summary, if it was taken on the
    current prefill sources (else None)."""
    path = os.path.join(ROOT, "profiles", "prefill_%s.md" % workload.replace("prefill_", "", 1))
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    s = re.search(r"prefill_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != code_hash(PREFILL_SOURCES):
        return None
    return int(m.group(1))


def run_prefill(args, name, world, rank, local_rank, K, W, full=True):
    """One prefill workload: K timed steps after W warm-up steps.  full: also the end-to-end
    leg from host memory and the oracle on the host."""
    import torch
    import paged_kv_cache_159_gb300 as pkv

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = workloads.PREFILL_WORKLOADS[name]
    d = workloads.draw_prefill(w, dev)
    Hq, Hkv, D = w.num_q_heads, w.num_kv_heads, w.head_dim
    T = int(d.cu_q[-1])
    fp8 = w.kv_dtype == "fp8"
    kc, vc = d.key_cache, d.value_cache
    if fp8:
        # an E4M3 pool, per-tensor scales amax / 448 over the bf16 history and chunks
        ks = float(np.float32(max(kc.float().abs().max().item(), d.k_chunk.float().abs().max().item()))
                   / np.float32(448.0))
        vs = float(np.float32(max(vc.float().abs().max().item(), d.v_chunk.float().abs().max().item()))
                   / np.float32(448.0))
        pool = pkv.Pool(d.num_blocks, Hkv, D, pkv.KV_FP8E4M3, ks, vs, d.free_order)
    else:
        pool = pkv.Pool(d.num_blocks, Hkv, D, free_order=d.free_order)
    pool.attach_device(local_rank)
    tables = pool.build_block_tables(d.seq_lens, d.max_blocks)
    slots = pkv.slot_mapping_chunks(tables, d.seq_lens, d.cu_q)
    if fp8:
        # the history (every position but the chunks') encoded into the pool by kv_append
        hist = np.setdiff1d(pkv.slot_mapping_all(tables, d.seq_lens), slots)
        hs = torch.from_numpy(hist).to(dev)
        k8 = torch.zeros(kc.shape, dtype=torch.uint8, device=dev)
        v8 = torch.zeros(vc.shape, dtype=torch.uint8, device=dev)
        for i in range(0, len(hist), 1 << 16):
            h = hs[i:i + (1 << 16)]
            pkv.kv_append(pool, kc[h // 16, :, h % 16, :].contiguous(), vc[h // 16, :, h % 16, :].contiguous(),
                          h, k8, v8)
        torch.cuda.synchronize()
        kc, vc = k8, v8
    plan_h, grid = pkv.prefill_plan(pool, d.cu_q, d.seq_lens, Hq, d.max_blocks)
    plan = torch.from_numpy(plan_h).to(dev)
    bt = torch.from_numpy(tables).to(dev)
    sm = torch.from_numpy(slots).to(dev)
    out = torch.empty_like(d.q)
    flops = _prefill_flops(d, Hq, D)
    stream = torch.cuda.Stream(device=dev)
    flush_buf = torch.ones(2 * torch.cuda.get_device_properties(dev).L2_cache_size // 4,
                           dtype=torch.int32, device=dev)
    flush_out = torch.empty((), dtype=torch.int64, device=dev)

    def step(s=None):
        pkv.kv_append(pool, d.k_chunk, d.v_chunk, sm, kc, vc, stream=s)
        mids_rec(s)
        pkv.paged_prefill(pool, d.q, kc, vc, bt, w.scale, plan, grid, out, stream=s)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    cur = [0]

    def mids_rec(s):
        mids[cur[0]].record(s)

    with torch.cuda.stream(stream):
        for i in range(W):
            cur[0] = i % K
            torch.sum(flush_buf, dim=0, out=flush_out)
            step(stream)
    stream.synchronize()
    st, bits = pool.get_device_error(stream)
    if st != pkv.OK:
        raise RuntimeError("device error in warm-up: %d bits %#x" % (st, bits))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for i in range(K):
                cur[0] = i
                torch.sum(flush_buf, dim=0, out=flush_out)
                starts[i].record(stream)
                step(stream)
                ends[i].record(stream)
        stream.synchronize()
        wall = time.perf_counter() - t0
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    total = float(sum(starts[i].elapsed_time(ends[i]) * 1e-3 for i in range(K)))
    pre_mean = float(sum(mids[i].elapsed_time(ends[i]) * 1e-3 for i in range(K)) / K)
    st, bits = pool.get_device_error(stream)
    if st != pkv.OK:
        raise RuntimeError("device error in the timed region: %d bits %#x" % (st, bits))

    def e2e_leg():
        # end to end: the step's inputs from pinned host memory, the output back, every step.
        # The batch is cut into groups of whole sequences, each with its own host plan; group
        # i+1's upload overlaps group i's kv_append + prefill and group i-1's download (three
        # streams).  Rows do not depend on the batch around them, so the output is the same.
        pin = lambda t: t.detach().cpu().pin_memory()
        ref_out = out.detach().cpu()
        B = w.batch
        NC = min(4, B)
        groups = []
        for c in range(NC):
            b0, b1 = c * B // NC, (c + 1) * B // NC
            r0, r1 = int(d.cu_q[b0]), int(d.cu_q[b1])
            cu = (d.cu_q[b0:b1 + 1] - d.cu_q[b0]).astype(np.int32)
            plan_c, grid_c = pkv.prefill_plan(pool, cu, d.seq_lens[b0:b1], Hq, d.max_blocks)
            groups.append(dict(
                rows=(r0, r1), bts=(b0, b1), grid=grid_c,
                hq=pin(d.q[r0:r1]), hk=pin(d.k_chunk[r0:r1]), hv=pin(d.v_chunk[r0:r1]), hbt=pin(bt[b0:b1]),
                hsm=pin(sm[r0:r1]), hplan=torch.from_numpy(plan_c).pin_memory(),
                dplan=torch.empty(plan_c.shape, dtype=torch.uint8, device=dev),
                hout=torch.empty((r1 - r0,) + tuple(out.shape[1:]), dtype=out.dtype).pin_memory()))
        h2d = sum(x.numel() * x.element_size() for g in groups for x in (g["hq"], g["hk"], g["hv"], g["hbt"], g["hsm"], g["hplan"]))
        d2h = sum(g["hout"].numel() * g["hout"].element_size() for g in groups)
        s_up, s_run, s_down = (torch.cuda.Stream(device=dev) for _ in range(3))
        ee = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev_in = [torch.cuda.Event() for _ in groups]
        ev_run = [torch.cuda.Event() for _ in groups]
        e2e_t = []
        for i in range(max(5, min(K, 100)) + 3):
            torch.sum(flush_buf, dim=0, out=flush_out)
            torch.cuda.synchronize()
            ee[0].record(s_up)
            for g, ei, er in zip(groups, ev_in, ev_run):
                (r0, r1), (b0, b1) = g["rows"], g["bts"]
                with torch.cuda.stream(s_up):
                    for dst, src in ((d.q[r0:r1], g["hq"]), (d.k_chunk[r0:r1], g["hk"]), (d.v_chunk[r0:r1], g["hv"]),
                                     (bt[b0:b1], g["hbt"]), (sm[r0:r1], g["hsm"]), (g["dplan"], g["hplan"])):
                        dst.copy_(src, non_blocking=True)
                    ei.record(s_up)
                s_run.wait_event(ei)
                pkv.kv_append(pool, d.k_chunk[r0:r1], d.v_chunk[r0:r1], sm[r0:r1], kc, vc, stream=s_run)
                pkv.paged_prefill(pool, d.q[r0:r1], kc, vc, bt[b0:b1], w.scale, g["dplan"], g["grid"], out[r0:r1],
                                  stream=s_run)
                er.record(s_run)
                s_down.wait_event(er)
                with torch.cuda.stream(s_down):
                    g["hout"].copy_(out[r0:r1], non_blocking=True)
            ee[1].record(s_down)
            ee[1].synchronize()
            if i >= 3:
                e2e_t.append(ee[0].elapsed_time(ee[1]) * 1e-3)
        for g in groups:                                    # the grouped step gives the same bits
            r0, r1 = g["rows"]
            if not torch.equal(g["hout"].view(torch.int16), ref_out[r0:r1].view(torch.int16)):
                raise RuntimeError("grouped end-to-end prefill output differs from the single launch")
        e2e_step = float(statistics.median(e2e_t))
        api = ("kv_append + paged_prefill per group of %d sequences (%d groups, own plans); uploads, "
               "kernels and downloads on three streams, overlapped across groups" % (B // NC, NC))
        return e2e_step, h2d, d2h, api

    e2e_step = h2d = d2h = None
    if full:
        e2e_step, h2d, d2h, e2e_api = e2e_leg()
    if world > 1:
        total, pre_mean = reduce_max_over_ranks([total, pre_mean], dev)
        if e2e_step is not None:
            (e2e_step,) = reduce_max_over_ranks([e2e_step], dev)
    peak, peak_src = _tensor_peak()
    value = world * flops * K / total / 1e12
    achieved = flops / pre_mean / 1e12
    traffic = _prefill_traffic(w.name)
    # algorithmic bytes of one prefill launch: K and V of every position, q and out of every
    # packed row, the tables
    alg_bytes = (int(d.seq_lens.astype(np.int64).sum()) * Hkv * D * (1 if fp8 else 2) * 2 + T * Hq * D * 2 * 2
                 + w.batch * d.max_blocks * 4)
    if not full:
        return {"value": round(value, 2), "unit": "TFLOP/s", "step": "kv_append + paged_prefill (tcgen05)",
                "ms_per_step": round(total / K * 1e3, 5), "kernel_us": round(pre_mean * 1e6, 2),
                "frac": round(achieved / peak, 4), "achieved": round(achieved, 2), "flops_per_launch": flops,
                "bytes_per_launch": alg_bytes, "traffic": traffic,
                "traffic_ratio": round(traffic / alg_bytes, 3) if traffic else None,
                "kernel": "prefill_kernel<%d%s>" % (D, ", fp8" if fp8 else ""), "steps": K, "warmup": W, "gpu_launches": 2 * K}
    res = {
        "metric": PREFILL_METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(total / K * 1e3, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": "%s: %d sequences, chunk %s, context %s, q heads %d / kv heads %d, head_dim %d, "
                        "block 16 (%d rows, %d causal key visits)" % (
                            w.name, w.batch, "U{1..%d}" % w.chunk if w.ragged else w.chunk,
                            ("U{0..%d}" % w.context) if w.context else "0", Hq, Hkv, D, T,
                            flops // (4 * Hq * D)),
            "step": "kv_append of the chunks + paged_prefill (tcgen05), plan made once on the host",
            "grid": grid, "parallelism": "replicas",
            "l2": "flushed between steps (read of a 2x L2 buffer)",
            "timing": "CUDA events around each step on the launch stream; flush outside them",
        },
        "query_tokens_per_s": round(world * T * K / total, 1),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "prefill_kernel<%d%s>" % (D, ", fp8" if fp8 else ""), "bytes_per_launch": alg_bytes,
                     "flops_per_launch": flops, "peak_source": peak_src},
        "e2e": {"value": round(world * flops / e2e_step / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e2e_step * 1e3, 4), "api": e2e_api},
        "gpu_launches": 2 * K,
        "clocks": clk.summary(),
        "wall_s_timed_region": round(wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        tf, sec, nrows, threads = _prefill_oracle_sample(w)
        res["cpu_baseline"] = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": int(threads), "kind": "oracle",
                               "sample": "the last %d rows of sequence 0, fp64, %.2f s" % (nrows, sec)}
    return res


def run_prefill_reference(args):
    w = workloads.PREFILL_WORKLOADS[args.workload]
    t = []
    for i in range(args.warmup + args.steps):
        tf, sec, nrows, threads = _prefill_oracle_sample(w, nrows=8)
        if i >= args.warmup:
            t.append(sec)
    total = float(sum(t))
    d = workloads.draw_prefill(w, "cpu")
    L = int(d.seq_lens[0])
    flops = 4 * w.num_q_heads * w.head_dim * sum(range(L - 8 + 1, L + 1))
    value = flops * args.steps / total / 1e12
    return {
        "impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "parallelism": "host threads",
                   "sample": "the last 8 rows of sequence 0 per step"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": "the last 8 rows of sequence 0 per step, %d steps" % args.steps},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


OTHER_CONFIGS = ("ragged", "llama3_70b_long", "qwen25_7b_prefix", "qwen25_7b_prefix_fp8",
                 "qwen25_7b_prefix_cow", "llama3_8b_32l", "prefill_llama3_8b", "chunked_prefill_llama3_8b",
                 "chunked_prefill_llama3_8b_fp8")


def run_other_configs(args, world, rank, local_rank):
    """Every other workload, timed in the same process after the headline: a compact line
    each (value, roofline fraction, traffic ratio, ms per step), and the clocks seen while
    they ran."""
    import gc
    import torch
    out = {}
    with ClockSampler(local_rank) as clk:
        for name in OTHER_CONFIGS:
            run = run_prefill if name in workloads.PREFILL_WORKLOADS else run_decode
            out[name] = run(args, name, world, rank, local_rank, args.other_steps, 5, full=False)
            gc.collect()
            torch.cuda.empty_cache()
    out["clocks"] = clk.summary()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(workloads.WORKLOADS) + sorted(workloads.PREFILL_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-seqs", type=int, default=64)
    ap.add_argument("--separate-append", action="store_true",
                    help="time kv_append and decode as two launches instead of decode_step")
    ap.add_argument("--opts", default="", help='decode knobs as JSON, e.g. {"warps_per_cta": 8}')
    ap.add_argument("--no-other-configs", action="store_true",
                    help="time only --workload (the default run also times every other workload)")
    ap.add_argument("--other-steps", type=int, default=30, help="timed steps of each other workload")
    ap.add_argument("--steady-steps", type=int, default=8000,
                    help="steps of the headline's steady repeat (clock samples under load); 0: none")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local_rank = _dist_env()
    if args.impl == "reference":
        if rank == 0:
            ref = run_prefill_reference if args.workload in workloads.PREFILL_WORKLOADS else run_reference
            print(json.dumps(ref(args)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run = run_prefill if args.workload in workloads.PREFILL_WORKLOADS else run_decode
        res = run(args, args.workload, world, rank, local_rank, args.steps, args.warmup, full=True)
        if args.workload == DEFAULT_WORKLOAD and not args.no_other_configs:
            res["other_configs"] = run_other_configs(args, world, rank, local_rank)
        if rank == 0:
            print(json.dumps(res), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
