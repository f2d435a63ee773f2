"""Benchmark of the UltraQuant FP4 KV-cache path on GB300.

Workload (per GPU): 64K-context decode, batch 8, 8 KV heads, 64 query heads,
head_dim 128, page size 16, shuffled pages.  Setup (untimed) quantize-appends
32768 tokens per sequence; the prefill-append of 32768 more tokens per
sequence is timed on its own (quantize GB/s); then one step = append one new
token per sequence + decode attention of one query token per sequence at
context 65536+i, straight from the packed cache.  value = decode tokens/s
(sequences x steps / time), whole job over all ranks.

--impl reference runs the CPU oracle (the plain C reference this library is
tested against) on a bounded sample of the same workload.

Output: one JSON line on rank 0.
"""
import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

B, HKV, HQ, D, PS = 8, 8, 64, 128, 16
CTX0, APPEND = 32768, 32768
FP4_BYTES_PER_TOKEN_HEAD = 136   # K and V: 64 code bytes + 4 scale bytes each
FP8_BYTES_PER_TOKEN_HEAD = 256
BF16_BYTES_PER_TOKEN_HEAD = 512
PF_CHUNK = 128                   # prefill chunk per sequence in the prefill measurement
REPEAT_S = 0.5                   # each timed region repeats its K steps until it lasts this long
MAX_REPEATS = 400
METRIC = "decode tokens/s at 64K ctx (KV-read GB/s and quantize GB/s reported)"
WORKLOAD = "append64k: B8 Hkv8 Hq64 D128 ps16, 32768 cached + 32768 appended tokens/seq, then decode steps"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _rank_seed(rank: int) -> int:
    """Seed of rank `rank`'s own batch of sequences (weak scaling: every rank a different batch)."""
    return 1005 + 7919 * rank


def _max_over_ranks(x: float, ws: int, device) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    if ws <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _job_throughput(ws: int, seqs_per_rank: int, steps: int, total_s: float) -> float:
    """Decode tokens/s of the whole job: every rank decodes its own sequences each step."""
    return ws * seqs_per_rank * steps / total_s


def _tensor_peak():
    """Measured dense bf16 tensor rate (TFLOP/s), or the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class Clocks:
    """SM clock and clock-event-reason sampler for the timed region.

    Polls NVML (libnvidia-ml, read-only queries) from a thread every 2 ms, so
    a timed region of a few tens of milliseconds still gets a dozen samples;
    falls back to `nvidia-smi -lms 100` where the library cannot be loaded."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # clock event reason bits of the NVML API
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40}

    def __init__(self, gpu_index, pci_bus_id=None):
        self.gpu = gpu_index
        self.p = None
        self.nv = None
        self.samples = []
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                # NVML numbers all GPUs of the machine; the PCI bus id names the one CUDA uses
                ok = pci_bus_id is not None and \
                    nv.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(h)) == 0
                if ok or nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(h)) == 0:
                    self.nv, self.h, self.ct = nv, h, ctypes
        except Exception:
            self.nv = None

    def _read(self):
        ct, nv = self.ct, self.nv
        mhz, mx, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if nv.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz)) != 0:  # 1 = SM clock
            return None
        nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ct.byref(mx))
        fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or nv.nvmlDeviceGetCurrentClocksThrottleReasons
        fn(self.h, ct.byref(rs))
        return mhz.value, mx.value, rs.value

    def start(self):
        self.samples = []
        if self.nv is not None:
            import threading
            self.stop_ev = threading.Event()

            def run():
                while not self.stop_ev.is_set():
                    r = self._read()
                    if r is not None:
                        self.samples.append(r)
                    time.sleep(0.002)
            self.th = threading.Thread(target=run, daemon=True)
            self.th.start()
            t0 = time.time()
            while not self.samples and time.time() - t0 < 1.0:
                time.sleep(0.001)
            return
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None

    def stop(self):
        if self.nv is not None:
            self.stop_ev.set()
            self.th.join(timeout=5)
            sm = [s[0] for s in self.samples]
            reasons = sorted(n for n, bit in self.BITS.items() if any(s[2] & bit for s in self.samples))
            return {"sm_mhz": float(np.median(sm)) if sm else None,
                    "sm_max_mhz": float(self.samples[-1][1]) if sm else None, "reasons": reasons,
                    "samples": len(sm), "source": "nvml, 2 ms"}
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except Exception:
            self.p.kill()
            out = ""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi, 100 ms"}


def _pci_bus_id(dev):
    """'dddddddd:bb:dd.0' of a CUDA device, or None where torch does not report it."""
    pr = torch.cuda.get_device_properties(dev)
    try:
        return "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
    except AttributeError:
        return None


def _cpu_baseline(w):
    """The oracle, as it stands, on this host's cores.  Decode: (sequence, kv
    head) pairs of the 64K workload (8 query heads each) spread over one thread
    per core -- ceil(cores / 8) sequences, so every core has a pair -- and one
    pair on one thread.  Quantize: the oracle's append of a token range of the
    workload, chunked over one thread per core, and on one thread.  The C calls
    run outside the interpreter lock."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    cores = os.cpu_count() or 1
    L = CTX0 + APPEND
    G = HQ // HKV
    to16 = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    n_seq = (cores + HKV - 1) // HKV
    bt = np.arange(L // PS, dtype=np.int32)[None]
    sl = np.array([L], np.int32)
    pairs = []
    for seq in range(n_seq):
        k, v = w.kv(seq, 0, L, device="cpu")
        q = to16(w.q(0, device="cpu")[seq:seq + 1])
        for h in range(HKV):  # one single-head cache per (sequence, kv head), its G query heads
            c = oracle.Cache(oracle.KIND_FP4, L // PS, 1, PS, D)
            c.append(to16(k[:, h:h + 1]), to16(v[:, h:h + 1]), np.arange(L))
            pairs.append((c, np.ascontiguousarray(q[:, h * G:(h + 1) * G])))
    run = lambda cq: cq[0].decode(cq[1], bt, sl)
    t0 = time.perf_counter()
    run(pairs[0])
    dt1 = time.perf_counter() - t0
    with ThreadPoolExecutor(max_workers=cores) as ex:
        t0 = time.perf_counter()
        list(ex.map(run, pairs))
        dtn = time.perf_counter() - t0
    # quantize leg: T tokens x 8 kv heads of sequence 0, bf16 in, FP4 out
    T = 8192
    k, v = w.kv(0, 0, T, device="cpu")
    k16, v16 = to16(k), to16(v)
    qbytes = T * HKV * (2 * D * 2 + FP4_BYTES_PER_TOKEN_HEAD) + T * 8
    c1 = oracle.Cache(oracle.KIND_FP4, T // PS, HKV, PS, D)
    t0 = time.perf_counter()
    c1.append(k16, v16, np.arange(T))
    qt1 = time.perf_counter() - t0
    chunk = (T + cores - 1) // cores
    chunks = [(i, min(T, i + chunk)) for i in range(0, T, chunk)]
    cn = oracle.Cache(oracle.KIND_FP4, T // PS, HKV, PS, D)
    with ThreadPoolExecutor(max_workers=cores) as ex:
        t0 = time.perf_counter()
        list(ex.map(lambda r: cn.append(k16[r[0]:r[1]], v16[r[0]:r[1]], np.arange(r[0], r[1])), chunks))
        qtn = time.perf_counter() - t0
    return {"value": n_seq / dtn, "unit": "decode tokens/s", "cores": cores, "kind": "oracle",
            "sample": "%d sequences x 8 kv heads (8 query heads each) at context %d, FP4 cache, fp64 attention, "
                      "C oracle, one thread per (sequence, kv head) on %d threads: %.2f s; one pair on one "
                      "thread: %.2f s; quantize-append of %d tokens x 8 kv heads: %.2f s on %d threads, "
                      "%.2f s on one" % (n_seq, L, cores, dtn, dt1, T, qtn, cores, qt1),
            "single_thread": {"value": 1.0 / (dt1 * HKV), "unit": "decode tokens/s", "cores": 1},
            "quantize": {"GB_per_s": qbytes / qtn / 1e9, "cores": cores,
                         "single_thread_GB_per_s": qbytes / qt1 / 1e9}}


def run_reference(args):
    """The oracle (this repository's plain C reference) on the same workload: the decode of
    kv head 0 of sequence 0 (its 8 query heads) over the 64K context.  The oracle's time is
    linear in the context, so each timed step decodes a prefix of the context sized to keep
    the whole --steps/--warmup run within a few minutes (calibrated on one full-context
    decode), and the value is scaled to the full context."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import workloads
    w = workloads.make("append64k", seq_lens=[CTX0 + APPEND] * B, extra_tokens=16)
    import oracle
    L = CTX0 + APPEND
    to16 = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    k, v = w.kv(0, 0, L, device="cpu")
    oc = oracle.Cache(oracle.KIND_FP4, L // PS, 1, PS, D)
    oc.append(to16(k[:, :1]), to16(v[:, :1]), np.arange(L))   # kv head 0 of sequence 0
    bt = np.arange(L // PS, dtype=np.int32)[None]
    q = to16(w.q(0, device="cpu")[0:1, :HQ // HKV])           # its 8 query heads
    t0 = time.perf_counter()
    oc.decode(q, bt, np.array([L], np.int32))
    t_full = time.perf_counter() - t0
    budget = 150.0  # seconds for warm-up and timed steps together
    Ls = int(min(L, max(PS, L * budget / (max(1, args.steps + args.warmup) * max(t_full, 1e-6)))))
    Ls -= Ls % PS
    sl = np.array([Ls], np.int32)
    for _ in range(args.warmup):
        oc.decode(q, bt, sl)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oc.decode(q, bt, sl)
    dt = time.perf_counter() - t0
    per = dt / args.steps * (L / Ls)  # one full-context step
    value = (1.0 / HKV) / per   # one step decodes 1/8 of one sequence's token
    sample = ("seq 0, kv head 0, 8 query heads; each step over the first %d of the %d context tokens, "
              "scaled to the full context (one full-context decode took %.3f s)" % (Ls, L, t_full))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "decode tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": value, "unit": "decode tokens/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "decode tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _event_pair():
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def run_uq(args):
    ws, rank, local = _dist()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import ue8m0_kv_cache_gb300 as uq
    import workloads

    steps, warmup = args.steps, args.warmup
    extra = steps + warmup + 8
    # Each rank holds its own batch of 8 sequences (weak scaling, no collective on the data path).
    w = workloads.make("append64k", seq_lens=[CTX0 + APPEND] * B, extra_tokens=extra, seed=_rank_seed(rank))
    stream = torch.cuda.current_stream()
    caches = {"fp4": uq.KVCache(uq.FP4_UE8M0, w.num_pages, HKV, PS, D, device=dev)}
    if not args.no_anchors:
        caches["fp8"] = uq.KVCache(uq.FP8_E4M3, w.num_pages, HKV, PS, D, device=dev)
        caches["bf16"] = uq.KVCache(uq.BF16, w.num_pages, HKV, PS, D, device=dev)
        caches["tq4"] = uq.KVCache(uq.TQ4, w.num_pages, HKV, PS, D, device=dev)

    # ---- setup: the cached 32768 tokens per sequence (untimed)
    for b in range(B):
        for t0 in range(0, CTX0, 8192):
            k, v = w.kv(b, t0, 8192, device=dev)
            sl = torch.from_numpy(w.slots(b, t0, 8192)).to(dev)
            for c in caches.values():
                uq.uq_quantize_append(k, v, sl, c)
    # ---- the prefill-append of 32768 more tokens per sequence: inputs resident, timed alone
    ks, vs, ss = [], [], []
    for b in range(B):
        k, v = w.kv(b, CTX0, APPEND, device=dev)
        ks.append(k)
        vs.append(v)
        ss.append(torch.from_numpy(w.slots(b, CTX0, APPEND)).to(dev))
    kA, vA, sA = torch.cat(ks), torch.cat(vs), torch.cat(ss)
    del ks, vs, ss
    for c in list(caches.values())[1:]:
        uq.uq_quantize_append(kA, vA, sA, c)
    fp4 = caches["fp4"]
    l2_flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def time_append(cache):
        times = []
        for i in range(3 + 5):
            l2_flush.zero_()
            e0, e1 = _event_pair()
            e0.record(stream)
            uq.uq_quantize_append(kA, vA, sA, cache)
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                times.append(e0.elapsed_time(e1) * 1e-3)
        return float(np.median(times))

    n_th = B * APPEND * HKV
    q_in, q_out = n_th * 2 * D * 2, n_th * FP4_BYTES_PER_TOKEN_HEAD + B * APPEND * 8
    q_t = time_append(fp4)
    hbm0, _ = _peaks()
    quantize = {"GB_per_s": (q_in + q_out) / q_t / 1e9, "ms": q_t * 1e3, "tokens": B * APPEND,
                "bytes_in": q_in, "bytes_out": q_out, "launches": 1,
                "frac": (q_in + q_out) / q_t / 1e9 / hbm0, "peak": hbm0}
    tq4_quantize = None
    if "tq4" in caches:  # the codebook variant writes the same 136 B per token-head
        tq_t = time_append(caches["tq4"])
        tq4_quantize = {"GB_per_s": (q_in + q_out) / tq_t / 1e9, "ms": tq_t * 1e3,
                        "frac": (q_in + q_out) / tq_t / 1e9 / hbm0}
    del kA, vA, sA, l2_flush
    assert uq.uq_check_device_status() == 0

    # ---- decode steps: per step one new token per sequence is appended, then decoded
    bt = torch.from_numpy(w.block_table).to(dev)
    L0 = CTX0 + APPEND
    n_new = steps + warmup
    kv_new = [w.kv(b, L0, n_new, device=dev) for b in range(B)]          # [n_new][Hkv][D] per sequence
    k_all = torch.stack([kv[0] for kv in kv_new], 1).contiguous()        # [n_new][B][Hkv][D]
    v_all = torch.stack([kv[1] for kv in kv_new], 1).contiguous()
    s_all = torch.from_numpy(np.stack([w.slots(b, L0, n_new) for b in range(B)], 1).copy()).to(dev)
    newk = [k_all[s] for s in range(n_new)]
    newv = [v_all[s] for s in range(n_new)]
    news = [s_all[s] for s in range(n_new)]
    q_pool = [w.q(1 + s, device=dev) for s in range(32)]
    qs = [q_pool[s % 32] for s in range(n_new)]
    del kv_new
    lens = [torch.full((B,), L0 + s + 1, dtype=torch.int32, device=dev) for s in range(n_new)]
    out = torch.empty((B, HQ, D), dtype=torch.float32, device=dev)
    wsp = uq.workspace(B, HQ, HKV, D, dev)
    decode_fn = {"fp4": uq.uq_decode_attention, "fp8": uq.uq_decode_attention_fp8,
                 "bf16": uq.uq_decode_attention_bf16, "tq4": uq.uq_decode_attention_tq4}

    def decode_loop(name, count, offset, timed_decode):
        c = caches[name]
        for s in range(offset, offset + count):
            if name != "fp4":
                uq.uq_quantize_append(newk[s], newv[s], news[s], c)
            if timed_decode is not None:
                e0, e1 = _event_pair()
                e0.record(stream)
            if name == "fp4":  # the step's new tokens are quantised inside the decode launch
                uq.uq_decode_attention_append(qs[s], newk[s], newv[s], news[s], c, bt, lens[s],
                                              out=out, workspace=wsp)
            else:
                decode_fn[name](qs[s], c, bt, lens[s], out=out, workspace=wsp)
            if timed_decode is not None:
                e1.record(stream)
                timed_decode.append((e0, e1))

    def timed(name, clocks=None):
        """W warm-up steps, then R repeats of exactly the K timed steps (each repeat
        replays the same K steps: the same new tokens into the same slots at the
        same contexts, so every repeat does identical work), R chosen so the timed
        region lasts >= REPEAT_S.  Returns (median repeat s, median decode launch s,
        repeat times, clocks)."""
        decode_loop(name, warmup, 0, None)
        torch.cuda.synchronize()
        t0, t1 = _event_pair()  # one untimed repeat sizes R
        t0.record(stream)
        decode_loop(name, steps, warmup, None)
        t1.record(stream)
        torch.cuda.synchronize()
        reps = int(min(MAX_REPEATS, max(1, np.ceil(REPEAT_S / max(t0.elapsed_time(t1) * 1e-3, 1e-6)))))
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        if clocks:
            clocks.start()
        ev, rep_ev = [], []
        for _ in range(reps):
            r0, r1 = _event_pair()
            r0.record(stream)
            decode_loop(name, steps, warmup, ev)
            r1.record(stream)
            rep_ev.append((r0, r1))
        torch.cuda.synchronize()
        clk = clocks.stop() if clocks else None
        if ws > 1:
            torch.distributed.barrier()
        rep = [a.elapsed_time(b) * 1e-3 for a, b in rep_ev]
        dec = float(np.median([a.elapsed_time(b) for a, b in ev])) * 1e-3
        return float(np.median(rep)), dec, rep, clk

    clocks = Clocks(local if os.environ.get("CUDA_VISIBLE_DEVICES") is None else 0, _pci_bus_id(dev))
    rep_t, dec_t, rep_all, clk = timed("fp4", clocks)
    assert uq.uq_check_device_status() == 0
    total = _max_over_ranks(rep_t, ws, dev)  # one repeat of the K steps, slowest rank
    ctx_mean = L0 + warmup + (steps + 1) / 2.0
    kv_bytes = B * HKV * ctx_mean * FP4_BYTES_PER_TOKEN_HEAD
    hbm, peak_kind = _peaks()
    ms_per_step = total / steps * 1e3
    value = _job_throughput(ws, B, steps, total)
    achieved = kv_bytes / dec_t / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": _captured_traffic(B * HKV * ctx_mean), "peak_kind": peak_kind,
                "kernel": "uq_decode_attention_append (fused append + decode, then merge), FP4 cache",
                "algorithmic_bytes_per_launch": kv_bytes, "launch_ms": dec_t * 1e3,
                "launch_ms_stat": "median over %d launches" % (len(rep_all) * steps),
                "frac_of_nominal_8TBps": achieved / 8000.0}
    timing = {"repeats": len(rep_all), "steps_per_repeat": steps, "repeat_ms_median": rep_t * 1e3,
              "repeat_ms_min": min(rep_all) * 1e3, "repeat_ms_max": max(rep_all) * 1e3,
              "timed_region_s": float(sum(rep_all)),
              "note": "value and ms_per_step from the median repeat of the K steps; every repeat replays the same "
                      "K steps (same tokens, slots and contexts)"}

    anchors = {}
    for name, per in (("fp8", FP8_BYTES_PER_TOKEN_HEAD), ("bf16", BF16_BYTES_PER_TOKEN_HEAD),
                      ("tq4", FP4_BYTES_PER_TOKEN_HEAD)):
        if name not in caches:
            continue
        tt, dt, _, _ = timed(name)
        gbs = B * HKV * ctx_mean * per / dt / 1e9
        anchors[name] = {"decode_tokens_per_s": B * steps / tt, "ms_per_step": tt / steps * 1e3,
                         "decode_ms": dt * 1e3, "kv_GB_per_s": gbs, "frac": gbs / hbm}
        if name == "tq4":
            anchors[name]["quantize"] = tq4_quantize
    assert uq.uq_check_device_status() == 0

    # ---- chunked-prefill attention over the same FP4 cache: the last PF_CHUNK
    # tokens of every sequence attend causally to its 64K context
    prefill = None
    if not args.no_anchors:
        T = B * PF_CHUNK
        gq = torch.Generator(device=dev)
        gq.manual_seed(4242 + rank)
        qp = torch.randn((T, HQ, D), generator=gq, device=dev).to(torch.bfloat16)
        cu = torch.arange(0, T + 1, PF_CHUNK, dtype=torch.int32, device=dev)
        slp = torch.full((B,), L0, dtype=torch.int32, device=dev)
        wsp_p = torch.empty(max(16, uq.uq_prefill_workspace_bytes(T, B, HQ, HKV, D, bt.shape[1] * PS)),
                            dtype=torch.uint8, device=dev)
        outp = torch.empty((T, HQ, D), dtype=torch.float32, device=dev)
        times = []
        for i in range(3 + 3):
            e0, e1 = _event_pair()
            e0.record(stream)
            uq.uq_prefill_attention(qp, cu, fp4, bt, slp, out=outp, workspace=wsp_p)
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                times.append(e0.elapsed_time(e1) * 1e-3)
        pt = float(np.median(times))
        keys = B * HQ * sum(L0 - PF_CHUNK + i + 1 for i in range(PF_CHUNK))
        flops = 4.0 * D * keys  # QK^T and P.V, one multiply-add each per (query row, key, channel)
        tens_peak = _tensor_peak()
        prefill = {"chunk_tokens_per_seq": PF_CHUNK, "context": L0, "ms": pt * 1e3, "TFLOP_per_s": flops / pt / 1e12,
                   "query_tokens_per_s": T / pt, "tensor_peak_TFLOP_per_s": tens_peak,
                   "frac_of_tensor_peak": flops / pt / 1e12 / tens_peak,
                   "note": "QK^T: tcgen05 kind::mxf8f6f4 block-scaled (E4M3 query x E2M1 keys, UE8M0 key scales "
                           "in tensor memory), M 128 x N 64 tiles; P.V: tcgen05 kind::f16, twice (hi + lo parts of P)"}
        del qp, wsp_p, outp
    assert uq.uq_check_device_status() == 0

    # ---- end to end through the public API with host buffers: the same K steps (same
    # tokens, slots, contexts) with each step's inputs copied from pinned host memory and
    # its output read back, repeated like the device-timed region.  Each step's inputs
    # (q, new K, new V, slots) are one packed pinned buffer and one copy; the copies run
    # on a second stream into double-buffered device inputs and outputs, so step i+1's
    # inputs and step i-1's output move while step i decodes.
    n_e2e = min(steps, 200)
    idx = list(range(warmup, warmup + n_e2e))
    parts = [qs[0], newk[0], newv[0], news[0]]
    offs, tot = [], 0
    for t in parts:
        offs.append(tot)
        tot += (t.numel() * t.element_size() + 255) // 256 * 256

    def views(buf):
        return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, parts)]

    hin = []
    for s_ in idx:
        hb = torch.empty(tot, dtype=torch.uint8).pin_memory()
        for v_, src in zip(views(hb), (qs[s_], newk[s_], newv[s_], news[s_])):
            v_.copy_(src.cpu())
        hin.append(hb)
    hout = [torch.empty((B, HQ, D), dtype=torch.float32).pin_memory() for _ in range(2)]
    din = [torch.empty(tot, dtype=torch.uint8, device=dev) for _ in range(2)]
    dviews = [views(b_) for b_ in din]
    dout = [torch.empty((B, HQ, D), dtype=torch.float32, device=dev) for _ in range(2)]
    cstream = torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    h2d_done, dec_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def h2d(i):  # inputs of step i into buffer i % 2, once step i - 2 has read it
        with torch.cuda.stream(cstream):
            if i >= 2:
                cstream.wait_event(dec_done[i & 1])
            din[i & 1].copy_(hin[i], non_blocking=True)
            h2d_done[i & 1].record(cstream)

    def e2e_pass():
        cstream.wait_stream(stream)  # nothing of the previous pass still reads these buffers
        h2d(0)
        for i, s_ in enumerate(idx):
            k2 = i & 1
            if i + 1 < len(idx):
                h2d(i + 1)  # queued ahead of step i's read-back, so it runs while step i decodes
            stream.wait_event(h2d_done[k2])
            if i >= 2:
                stream.wait_event(d2h_done[k2])  # step i-2's output has been read back
            dq, dk, dv, dsl = dviews[k2]
            uq.uq_decode_attention_append(dq, dk, dv, dsl, fp4, bt, lens[s_], out=dout[k2], workspace=wsp)
            dec_done[k2].record(stream)
            with torch.cuda.stream(cstream):
                cstream.wait_event(dec_done[k2])
                hout[k2].copy_(dout[k2], non_blocking=True)
                d2h_done[k2].record(cstream)
        stream.wait_event(d2h_done[(len(idx) - 1) & 1])

    e2e_pass()
    torch.cuda.synchronize()
    e2e_rep = []
    for _ in range(len(rep_all)):
        t0, t1 = _event_pair()
        t0.record(stream)
        e2e_pass()
        t1.record(stream)
        e2e_rep.append((t0, t1))
    torch.cuda.synchronize()
    e2e_t = _max_over_ranks(float(np.median([a.elapsed_time(b) * 1e-3 for a, b in e2e_rep])), ws, dev)
    h2d = sum(t.numel() * t.element_size() for t in parts)
    e2e = {"value": ws * B * n_e2e / e2e_t, "unit": "decode tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": hout[0].numel() * 4, "steps": n_e2e, "repeats": len(e2e_rep),
           "stat": "median repeat",
           "pipeline": "one packed H2D copy per step and one D2H read on a second stream, double-buffered, "
                       "overlapping the neighbouring steps' decode"}
    assert uq.uq_check_device_status() == 0

    # ---- the mixed-length serving batch (B 64, seq_len ~ U[8192, 65536]), decode only
    mixed = None
    if not args.no_anchors:
        mixed = _mixed_decode(uq, dev, stream, steps, warmup, hbm, peak_kind)
    assert uq.uq_check_device_status() == 0

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        try:
            cpu = _cpu_baseline(w)
        except Exception as e:  # reported, not fatal
            cpu = {"error": repr(e)}
    line = {"metric": METRIC, "value": value, "unit": "decode tokens/s", "n_gpus": ws, "steps": steps,
            "warmup": warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e2m1/ue8m0 cache, f16 tensor-core MMA, f32 accumulate",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "context_mean": ctx_mean, "batch_per_gpu": B,
                       "parallelism": "replicas (weak scaling, no collective)" if ws > 1 else "single GPU",
                       "l2": "inputs larger than L2 (FP4 KV read %.0f MB per step)" % (kv_bytes / 1e6)},
            "kv_GB_per_s": achieved, "quantize": quantize, "anchors": anchors, "prefill": prefill, "roofline": roofline,
            "timing": timing, "mixed": mixed, "clocks": clk, "e2e": e2e,
            "gpu_launches": 2 * steps * len(rep_all), "cpu_baseline": cpu}
    print(json.dumps(line), flush=True)


def _mixed_decode(uq, dev, stream, steps, warmup, hbm, peak_kind):
    """Decode of the mixed-length serving batch: 64 sequences, 8 kv heads, 64 query
    heads, seq_len ~ U[8192, 65536] (seeded), 1% of tokens x8, shuffled pages.  The
    cache is filled untimed; each step decodes one query token per sequence (decode +
    merge launches); R repeats of K steps as the main line."""
    import workloads
    w = workloads.make("mixed")
    cache = uq.KVCache(uq.FP4_UE8M0, w.num_pages, w.Hkv, w.ps, w.D, device=dev)
    for b in range(w.B):
        for t0 in range(0, w.seq_lens[b], 8192):
            n = min(8192, w.seq_lens[b] - t0)
            k, v = w.kv(b, t0, n, device=dev)
            uq.uq_quantize_append(k, v, torch.from_numpy(w.slots(b, t0, n)).to(dev), cache)
    bt = torch.from_numpy(w.block_table).to(dev)
    sl = torch.tensor(w.seq_lens, dtype=torch.int32, device=dev)
    qs = [w.q(s, device=dev) for s in range(4)]
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device=dev)
    wsp = uq.workspace(w.B, w.Hq, w.Hkv, w.D, dev)

    def run(n, ev):
        for s in range(n):
            if ev is not None:
                e0, e1 = _event_pair()
                e0.record(stream)
            uq.uq_decode_attention(qs[s % 4], cache, bt, sl, out=out, workspace=wsp)
            if ev is not None:
                e1.record(stream)
                ev.append((e0, e1))

    run(warmup, None)
    torch.cuda.synchronize()
    t0, t1 = _event_pair()
    t0.record(stream)
    run(steps, None)
    t1.record(stream)
    torch.cuda.synchronize()
    reps = int(min(MAX_REPEATS, max(1, np.ceil(REPEAT_S / max(t0.elapsed_time(t1) * 1e-3, 1e-6)))))
    ev, rep = [], []
    for _ in range(reps):
        r0, r1 = _event_pair()
        r0.record(stream)
        run(steps, ev)
        r1.record(stream)
        rep.append((r0, r1))
    torch.cuda.synchronize()
    rt = float(np.median([a.elapsed_time(b) * 1e-3 for a, b in rep]))
    dt = float(np.median([a.elapsed_time(b) for a, b in ev])) * 1e-3
    kv = sum(w.seq_lens) * w.Hkv * FP4_BYTES_PER_TOKEN_HEAD
    res = {"workload": "mixed: B64 Hkv8 Hq64 D128 ps16, seq_len ~ U[8192, 65536] (%d tokens), 1%% of tokens x8"
                       % sum(w.seq_lens),
           "decode_tokens_per_s": w.B * steps / rt, "ms_per_step": rt / steps * 1e3, "launch_ms": dt * 1e3,
           "kv_GB_per_s": kv / dt / 1e9, "frac": kv / dt / 1e9 / hbm, "peak": hbm, "peak_kind": peak_kind,
           "repeats": reps, "l2": "inputs larger than L2 (%.2f GB per step)" % (kv / 1e9)}
    del cache, wsp
    return res


def decode_source_sha():
    """First 16 hex digits of the SHA-256 of the FP4 decode kernel's sources
    (the kernel file, then the header it shares with the tensor-memory decode)."""
    import hashlib
    h = hashlib.sha256()
    for name in ("uq_decode.cu", "uq_decode_common.cuh"):
        with open(os.path.join(ROOT, "ue8m0_kv_cache_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _captured_traffic(token_heads):
    """DRAM bytes (read + write) of one FP4 decode launch over `token_heads`
    token-heads, scaled from the ncu capture summarised in
    profiles/decode_fp4_traffic.json.  None when that capture is missing or was
    taken on a different version of the decode source."""
    try:
        with open(os.path.join(ROOT, "profiles", "decode_fp4_traffic.json")) as f:
            prof = json.load(f)
        sha = decode_source_sha()
    except (OSError, ValueError):
        return None
    if prof.get("source_sha256_16") != sha:
        return None
    return float(prof["dram_bytes_per_token_head"]) * token_heads


def run_decode_only(args):
    """Decode of one of the other workloads (tiny, gqa8k, mixed, prefix128k):
    the cache is filled untimed, then each step decodes one query token per
    sequence.  Used for per-workload numbers and for profiling."""
    ws, rank, local = _dist()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import ue8m0_kv_cache_gb300 as uq
    import workloads
    over = {}
    if args.batch > 0:
        base = workloads.make(args.workload)
        over = dict(B=args.batch, seq_lens=[base.seq_lens[b % base.B] for b in range(args.batch)])
    w = workloads.make(args.workload, **over)
    cache = uq.KVCache(uq.FP4_UE8M0, w.num_pages, w.Hkv, w.ps, w.D, device=dev)
    for b in range(w.B):
        start = w.shared_prefix if (b > 0 and w.shared_prefix) else 0
        for t0 in range(start, w.seq_lens[b], 8192):
            n = min(8192, w.seq_lens[b] - t0)
            k, v = w.kv(b, t0, n, device=dev)
            uq.uq_quantize_append(k, v, torch.from_numpy(w.slots(b, t0, n)).to(dev), cache)
    bt = torch.from_numpy(w.block_table).to(dev)
    sl = torch.tensor(w.seq_lens, dtype=torch.int32, device=dev)
    if args.kernel == "prefill":
        return _prefill_only(args, uq, w, cache, bt, sl, dev)
    if args.kernel == "cascade":
        return _cascade_only(args, uq, w, cache, bt, sl, dev)
    q = w.q(0, device=dev)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device=dev)
    wsp = uq.workspace(w.B, w.Hq, w.Hkv, w.D, dev)
    for _ in range(args.warmup):
        uq.uq_decode_attention(q, cache, bt, sl, out=out, workspace=wsp)
    torch.cuda.synchronize()
    t0, t1 = _event_pair()
    stream = torch.cuda.current_stream()
    t0.record(stream)
    for _ in range(args.steps):
        uq.uq_decode_attention(q, cache, bt, sl, out=out, workspace=wsp)
    t1.record(stream)
    torch.cuda.synchronize()
    assert uq.uq_check_device_status() == 0
    dt = t0.elapsed_time(t1) * 1e-3 / args.steps
    logical = sum(w.seq_lens) * w.Hkv * FP4_BYTES_PER_TOKEN_HEAD
    unique_tokens = sum(w.seq_lens) - (w.B - 1) * w.shared_prefix
    hbm, kind = _peaks()
    line = {"metric": "decode tokens/s (one attention layer)", "value": w.B / dt, "unit": "decode tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "dtype": "e2m1/ue8m0 cache", "data": "synthetic",
            "config": {"workload": args.workload, "B": w.B, "Hkv": w.Hkv, "Hq": w.Hq, "tokens": sum(w.seq_lens)},
            "kv_GB_per_s_logical": logical / dt / 1e9,
            "kv_GB_per_s_unique": unique_tokens * w.Hkv * FP4_BYTES_PER_TOKEN_HEAD / dt / 1e9,
            "frac_of_peak_logical": logical / dt / 1e9 / hbm, "peak": hbm, "peak_kind": kind,
            "gpu_launches": 2 * args.steps}
    print(json.dumps(line), flush=True)


def _prefill_only(args, uq, w, cache, bt, sl, dev):
    """Chunked-prefill attention on a filled cache: the last --chunk tokens of
    every sequence attend causally to the whole sequence."""
    n = min(args.chunk, min(w.seq_lens))
    T = w.B * n
    g = torch.Generator(device=dev)
    g.manual_seed(4242)
    q = torch.randn((T, w.Hq, w.D), generator=g, device=dev).to(torch.bfloat16)
    cu = torch.arange(0, T + 1, n, dtype=torch.int32, device=dev)
    wsp = torch.empty(max(16, uq.uq_prefill_workspace_bytes(T, w.B, w.Hq, w.Hkv, w.D, bt.shape[1] * w.ps)),
                      dtype=torch.uint8, device=dev)
    out = torch.empty((T, w.Hq, w.D), dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        uq.uq_prefill_attention(q, cu, cache, bt, sl, out=out, workspace=wsp)
    torch.cuda.synchronize()
    t0, t1 = _event_pair()
    stream = torch.cuda.current_stream()
    t0.record(stream)
    for _ in range(args.steps):
        uq.uq_prefill_attention(q, cu, cache, bt, sl, out=out, workspace=wsp)
    t1.record(stream)
    torch.cuda.synchronize()
    assert uq.uq_check_device_status() == 0
    dt = t0.elapsed_time(t1) * 1e-3 / args.steps
    keys = w.Hq * sum(L - n + i + 1 for L in w.seq_lens for i in range(n))
    flops = 4.0 * w.D * keys
    peak = _tensor_peak()
    line = {"metric": "chunked-prefill attention TFLOP/s", "value": flops / dt / 1e12, "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "dtype": "e2m1/ue8m0 cache; block-scaled e4m3 x e2m1 QK, f16 P.V",
            "data": "synthetic",
            "config": {"workload": args.workload, "B": w.B, "Hkv": w.Hkv, "Hq": w.Hq, "chunk": n,
                       "tokens": sum(w.seq_lens)},
            "tensor_peak_TFLOP_per_s": peak, "frac_of_tensor_peak": flops / dt / 1e12 / peak,
            "gpu_launches": 4 * args.steps}
    print(json.dumps(line), flush=True)


def _cascade_only(args, uq, w, cache, bt, sl, dev):
    """Cascade decode: all sequences form one group over the workload's shared
    prefix; the plain decode of the same step is timed beside it."""
    q = w.q(0, device=dev)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device=dev)
    cu = torch.tensor([0, w.B], dtype=torch.int32, device=dev)
    pre = torch.tensor([w.shared_prefix], dtype=torch.int32, device=dev)
    wsc = torch.empty(uq.uq_cascade_workspace_bytes(w.B, 1, w.Hq, w.Hkv, w.D, w.shared_prefix), dtype=torch.uint8,
                      device=dev)
    wsp = uq.workspace(w.B, w.Hq, w.Hkv, w.D, dev)
    stream = torch.cuda.current_stream()

    def timed(f):
        for _ in range(args.warmup):
            f()
        torch.cuda.synchronize()
        t0, t1 = _event_pair()
        t0.record(stream)
        for _ in range(args.steps):
            f()
        t1.record(stream)
        torch.cuda.synchronize()
        assert uq.uq_check_device_status() == 0
        return t0.elapsed_time(t1) * 1e-3 / args.steps

    dc = timed(lambda: uq.uq_cascade_decode_attention(q, cache, bt, sl, cu, pre, w.shared_prefix,
                                                      min_rows=args.min_rows, out=out, workspace=wsc))
    dp = timed(lambda: uq.uq_decode_attention(q, cache, bt, sl, out=out, workspace=wsp))
    logical = sum(w.seq_lens) * w.Hkv * FP4_BYTES_PER_TOKEN_HEAD
    unique = (sum(w.seq_lens) - (w.B - 1) * w.shared_prefix) * w.Hkv * FP4_BYTES_PER_TOKEN_HEAD
    hbm, kind = _peaks()
    line = {"metric": "cascade decode tokens/s (one attention layer)", "value": w.B / dc, "unit": "decode tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dc * 1e3,
            "higher_is_better": True, "dtype": "e2m1/ue8m0 cache", "data": "synthetic",
            "config": {"workload": args.workload, "B": w.B, "Hkv": w.Hkv, "Hq": w.Hq, "tokens": sum(w.seq_lens),
                       "shared_prefix": w.shared_prefix, "min_rows": args.min_rows},
            "plain_decode_ms": dp * 1e3, "speedup_vs_plain_decode": dp / dc,
            "kv_GB_per_s_unique": unique / dc / 1e9, "kv_GB_per_s_logical": logical / dc / 1e9,
            "frac_of_peak_unique": unique / dc / 1e9 / hbm, "peak": hbm, "peak_kind": kind,
            "gpu_launches": 5 * args.steps}
    print(json.dumps(line), flush=True)


def run_layers(args):
    """A decode step through every attention layer of an L-layer stack (B 8, Hkv 8, Hq 64, D 128, context
    --ctx): each layer appends the step's token and decodes.  The policy stack keeps the first and last two
    layers in BF16 and the rest in FP4; all-FP4 and all-FP8 stacks are timed beside it; steps replay one
    captured CUDA graph per stack (eager timed too for the policy stack)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import ue8m0_kv_cache_gb300 as uq
    import workloads
    from ue8m0_kv_cache_gb300.policy import LayeredKVCache, LayerPolicy, layered_workspace
    L = args.layers
    w = workloads.make("gqa8k", B=B, Hkv=HKV, Hq=HQ, D=D, ps=PS, seq_lens=[args.ctx] * B, seed=1006,
                       extra_tokens=args.steps + args.warmup + 16)
    stacks = {"policy_bf16_boundary2": LayerPolicy(L, boundary=2),
              "all_fp4": LayerPolicy(L, boundary=0),
              "all_fp8": LayerPolicy(L, boundary=0, inner=uq.FP8_E4M3)}
    caches = {k: LayeredKVCache(p, w.num_pages, HKV, PS, D, device=dev) for k, p in stacks.items()}
    for b in range(B):  # every layer holds the same values (timing does not depend on them)
        for t0 in range(0, args.ctx, 8192):
            n = min(8192, args.ctx - t0)
            k, v = w.kv(b, t0, n, device=dev)
            sl_b = torch.from_numpy(w.slots(b, t0, n)).to(dev)
            for lc in caches.values():
                for l in range(L):
                    lc.append(l, k, v, sl_b)
    torch.cuda.synchronize()
    bt = torch.from_numpy(w.block_table).to(dev)
    seq = torch.full((B,), args.ctx + 1, dtype=torch.int32, device=dev)
    slots = torch.from_numpy(np.array([w.slots(b, args.ctx, 1)[0] for b in range(B)])).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(77)
    q = [torch.randn((B, HQ, D), generator=g, device=dev).to(torch.bfloat16) for _ in range(L)]
    kn = [torch.randn((B, HKV, D), generator=g, device=dev).to(torch.bfloat16) for _ in range(L)]
    vn = [torch.randn((B, HKV, D), generator=g, device=dev).to(torch.bfloat16) for _ in range(L)]
    out = [torch.empty((B, HQ, D), dtype=torch.float32, device=dev) for _ in range(L)]
    wsp = layered_workspace(B, HQ, HKV, D, dev)
    stream = torch.cuda.current_stream()

    def timed(f):
        for _ in range(args.warmup):
            f()
        torch.cuda.synchronize()
        t0, t1 = _event_pair()
        t0.record(stream)
        for _ in range(args.steps):
            f()
        t1.record(stream)
        torch.cuda.synchronize()
        assert uq.uq_check_device_status() == 0
        return t0.elapsed_time(t1) * 1e-3 / args.steps

    res = {}
    pol = caches["policy_bf16_boundary2"]
    res["policy_eager_ms"] = 1e3 * timed(lambda: pol.decode_step(q, kn, vn, slots, bt, seq, out, wsp))
    for name, lc in caches.items():
        lc.capture_step(q, kn, vn, slots, bt, seq, out, wsp)
        res[name + "_graph_ms"] = 1e3 * timed(lc.replay)
        res[name + "_cache_GB"] = lc.nbytes() / 1e9
    dt = res["policy_bf16_boundary2_graph_ms"] * 1e-3
    line = {"metric": "decode tokens/s through all attention layers", "value": B / dt, "unit": "decode tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "dtype": "bf16 boundary layers, e2m1/ue8m0 inner layers", "data": "synthetic",
            "config": {"workload": "layers%d_ctx%d" % (L, args.ctx), "B": B, "Hkv": HKV, "Hq": HQ, "D": D,
                       "layers": L, "context": args.ctx},
            "stacks": res, "gpu_launches": args.steps * (2 * L + stacks["policy_bf16_boundary2"].count(uq.BF16))}
    print(json.dumps(line), flush=True)


def main():
    global REPEAT_S
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="uq", choices=["uq", "reference"])
    ap.add_argument("--no-anchors", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=None, choices=["append64k", "tiny", "gqa8k", "mixed", "prefix128k"],
                    help="default: prefix128k for --kernel cascade (the shared-prefix workload), else append64k")
    ap.add_argument("--kernel", default="decode", choices=["decode", "prefill", "cascade", "layers"],
                    help="with a workload other than append64k: what each step runs")
    ap.add_argument("--chunk", type=int, default=16, help="--kernel prefill: query tokens per sequence")
    ap.add_argument("--min-rows", type=int, default=0, help="--kernel cascade: min_rows of the cascade call")
    ap.add_argument("--batch", type=int, default=0, help="with a workload other than append64k: override B")
    ap.add_argument("--layers", type=int, default=32, help="--kernel layers: attention layers in the stack")
    ap.add_argument("--ctx", type=int, default=32768, help="--kernel layers: context per sequence")
    ap.add_argument("--repeat-s", type=float, default=REPEAT_S,
                    help="the K timed steps repeat until the timed region lasts this long (0: once)")
    args = ap.parse_args()
    if args.workload is None:
        args.workload = "prefix128k" if args.kernel == "cascade" else "append64k"
    args.warmup = max(args.warmup, 3)
    REPEAT_S = max(0.0, args.repeat_s)
    if args.impl == "reference":
        run_reference(args)
    elif args.kernel == "layers":
        run_layers(args)
    elif args.workload != "append64k" or args.kernel != "decode":
        run_decode_only(args)
    else:
        run_uq(args)


if __name__ == "__main__":
    main()
