"""Benchmark: fresh-session exact byte-level BPE encode on one GB300.

  python bench.py [--config C1..C5] [--gpus N] [--steps K] [--warmup W]
                  [--impl ours|reference] [--no-cpu-baseline]

Workloads (all synthetic and seeded; C3 is the default):
  C1  GPT-2 pattern, 1,000 merges; one 16 KiB string of code-like ASCII
  C2  GPT-2 pattern, 50,000 merges; one 1 MiB mixed text (code, CJK, accents,
      digit/whitespace runs)
  C3  cl100k-style pattern, 100,000 merges; one 1,000,000-character agentic
      session (fresh-session init)
  C4  cl100k-style, 100,000 merges; 64 sessions of log-uniform length
      (2 KiB .. 1 MiB, 15.0 MB in all) in one tok_encode_batch call
  C5  the 8 MiB adversarial text, encoded with the GPT-2 and the cl100k-style
      pattern (100,000 merges each): one step is both encodes

One step = the whole encode (UTF-8 decode, pre-tokenization, BPE, id
scatter) of every text of the workload, from device-resident input through
the device entry points (tok_encode_device / tok_encode_batch_device).
Before each timed step a 256 MiB buffer is written to flush L2 (every input
is smaller than L2); a second set of steps without the flush (vocabulary
tables and text L2-resident, as in a serving process) is reported as
`warm_l2`.  Steps are timed with CUDA events on the stream the kernels run
on; per-kernel times come from the library's own events around each kernel,
in a separate pass of the same flushed steps.  `e2e` times the host entry
points (tok_encode / tok_encode_batch) from pinned host memory into pinned
host memory, with the host clock.

With N > 1 (torchrun): C4 is split over the ranks (each encodes its share of
the 64 sessions in one batch call; strong scaling, the sessions are
independent so there is no collective); every other workload runs as one
replica per rank (a single text does not shard; weak scaling).  Rank 0
prints one JSON line with the max time over ranks.

--impl reference times the oracle (plain Python, one host core) on a bounded
sample of the same workload per step; rank 0 only.
"""
import argparse
import ctypes
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MB/s and ms per 1M chars, IDs bit-exact vs oracle; % of HBM roofline"
UNIT = "MB/s"
VOCABS = os.path.join(ROOT, "data", "vocabs")
GPT2, CL100K = 0, 1


# --- workloads ---------------------------------------------------------------

def _c1():
    import textgen
    return [textgen.code_ascii(16384, 1001)]


def _c2():
    import textgen
    return [textgen.mixed_c2(1 << 20, 1002)]


def _c3():
    import textgen
    return [textgen.agentic_session(1_000_000, 1003)]


def _c4():
    import textgen
    return textgen.session_batch(64, 1004)


def _c5():
    import textgen
    return [textgen.adversarial(8 << 20, 1005)]


CONFIGS = {
    "C1": {"workload": "GPT-2 pattern, 256 + 1,000 merges trained on a seeded 2 MiB code-like ASCII corpus; one "
                       "16,384-byte seeded string of code-like ASCII",
           "runs": [("gpt2_code_1k", GPT2)], "texts": _c1, "batch": False},
    "C2": {"workload": "GPT-2 pattern, 256 + 50,000 merges trained on a seeded 64 MiB corpus; one 1 MiB text: 80% "
                       "code-like ASCII, 10% CJK, 5% accented Latin, 5% digit/whitespace/newline runs",
           "runs": [("gpt2_mixed_50k", GPT2)], "texts": _c2, "batch": False},
    "C3": {"workload": "cl100k-style pattern, 256 + 100,000 merges trained on a seeded 64 MiB session corpus; one "
                       "1,000,000-character synthetic agentic session (fresh-session init)",
           "runs": [("cl100k_session_100k", CL100K)], "texts": _c3, "batch": False},
    "C4": {"workload": "cl100k-style pattern, 256 + 100,000 merges; a batch of 64 fresh synthetic agentic sessions, "
                       "lengths log-uniform 2 KiB to 1 MiB, in one tok_encode_batch call",
           "runs": [("cl100k_session_100k", CL100K)], "texts": _c4, "batch": True},
    "C5": {"workload": "adversarial 8 MiB text (100K-character whitespace runs, 200K-digit runs, a 1M-character "
                       "letter run, chained contractions, mixed CRLF/LF, every UTF-8 length class), encoded with "
                       "the GPT-2 and the cl100k-style pattern, 256 + 100,000 merges each",
           "runs": [("gpt2_session_100k", GPT2), ("cl100k_session_100k", CL100K)], "texts": _c5, "batch": False},
}

L2_NOTE = "flushed before every timed step (256 MiB write)"
ORACLE_SAMPLE_S = 10.0  # oracle seconds of the cpu_baseline leg (the sample is repeated up to this)


def config_line(name, texts_b, n_chars):
    """The `config` object of both arms (identical, so the lines compare)."""
    cfg = CONFIGS[name]
    return {"workload": cfg["workload"], "name": name, "bytes": sum(len(t) for t in texts_b), "chars": n_chars,
            "texts": len(texts_b), "patterns": ["gpt2" if p == GPT2 else "cl100k-style" for _, p in cfg["runs"]],
            "l2": L2_NOTE}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _sources_hash():
    """SHA-256 of the kernel sources, comments and whitespace removed (the
    DRAM counters stay valid across comment edits, not across code changes)."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_bpe_tokenization_utf_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".inc")):
            with open(os.path.join(csrc, f), encoding="utf-8", errors="replace") as fh:
                text = fh.read()
            text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
            text = re.sub(r"//[^\n]*", " ", text)
            text = " ".join(text.split())
            h.update(f.encode() + text.encode())
    return h.hexdigest()


def _traffic(config, kernel):
    """DRAM bytes per step of `kernel` on `config` from the committed ncu
    summary, if the kernel sources have not changed since it was taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("sources_sha256") != _sources_hash():
        return None
    e = d.get("configs", {}).get(config, {}).get(kernel)
    return e.get("bytes_per_step") if e else None


def host_cpu():
    """CPU model and core count of the host."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return {"cpu_model": model or platform.processor() or platform.machine(), "host_cores": os.cpu_count(),
            "arch": platform.machine()}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 20 ms, logged to a
    file while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        # the samples go to BENCH_CLOCKS_CSV when set (to keep them), else to
        # a scratch file; the JSON line carries their summary either way
        self.path = os.environ.get("BENCH_CLOCKS_CSV") or os.path.join(tempfile.gettempdir(),
                                                                        "bench_clocks_%d.csv" % os.getpid())

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "20", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.5)  # let the first samples arrive
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.rows = []
        if not self.proc:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        self.rows.append(parts)
        except Exception:
            pass

    def summary(self):
        rows = getattr(self, "rows", [])
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(r[1]) for r in rows) if v is not None]
        mx = [v for v in (num(r[2]) for r in rows) if v is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for k, nm in enumerate(names):
                if r[5 + k].lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# --- the oracle on the host cores --------------------------------------------

def _oracle_job(args):
    data, vocab_name, pattern = args
    from oracle.encode import encode
    from oracle.vocab import Vocab
    return len(encode(data, Vocab.load_merges(os.path.join(VOCABS, vocab_name + ".merges")), pattern))


def _windows(text, size, count):
    """`count` windows of about `size` characters of a text, spread over it."""
    if len(text) <= size:
        return [text] * count
    step = max(1, (len(text) - size) // max(1, count))
    return [text[(k * step) % (len(text) - size):][:size] for k in range(count)]


def reference_samples(name, texts, n):
    """(bytes, vocab name, pattern) of the oracle's n bounded samples of a
    workload: the whole text for C1, else 40,000-character windows (of the
    batch's sessions in turn for C4; alternating patterns for C5)."""
    cfg = CONFIGS[name]
    runs = cfg["runs"]
    out = []
    if name == "C1":
        return [(texts[0].encode(), runs[0][0], runs[0][1])] * n
    pool = texts if cfg["batch"] else [texts[0]]
    for k in range(n):
        t = pool[k % len(pool)]
        w = _windows(t, 40_000, n)[k]
        vname, pat = runs[k % len(runs)]
        out.append((w.encode(), vname, pat))
    return out


def cpu_baseline(name, texts_b, vocabs):
    """The oracle, as it stands, on a bounded sample of the workload on one
    host core; for C4 also over all host cores on the whole batch."""
    from oracle.encode import encode
    cfg = CONFIGS[name]
    cpu = host_cpu()
    if name == "C1":
        sample = [(texts_b[0], 0)]
        what = "the whole 16 KiB text"
    elif name == "C4":
        order = sorted(range(len(texts_b)), key=lambda k: len(texts_b[k]))
        pick, tot = [], 0
        for k in order:
            if tot > 1_500_000:
                break
            pick.append(k)
            tot += len(texts_b[k])
        sample = [(texts_b[k], 0) for k in pick]
        what = "the %d shortest sessions of the batch (%d bytes)" % (len(pick), tot)
    elif name == "C5":
        sample = [(texts_b[0][:1 << 20].decode("utf-8", "ignore").encode(), r) for r in range(len(cfg["runs"]))]
        what = "the first 1 MiB of the text under each pattern"
    else:
        sample = [(texts_b[0], 0)]
        what = "the whole text (%d bytes)" % len(texts_b[0])
    # the sample, repeated until at least ORACLE_SAMPLE_S seconds of oracle work
    t0 = time.perf_counter()
    nb, passes = 0, 0
    while passes == 0 or time.perf_counter() - t0 < ORACLE_SAMPLE_S:
        for data, r in sample:
            vname, pat = cfg["runs"][r]
            encode(data, vocabs[vname], pat)
            nb += len(data)
        passes += 1
    dt = time.perf_counter() - t0
    out = {"value": nb / dt / 1e6, "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": "%s, %d pass%s, single-threaded Python" % (what, passes, "" if passes == 1 else "es"),
           "seconds": dt, **cpu}
    if name == "C4":
        import multiprocessing as mp
        procs = os.cpu_count() or 1
        jobs = sorted([(t, cfg["runs"][0][0], cfg["runs"][0][1]) for t in texts_b], key=lambda j: -len(j[0]))
        with mp.get_context("spawn").Pool(procs) as pool:
            pool.map(_oracle_job, jobs[:procs], chunksize=1)  # workers up, vocabulary code loaded
            t0 = time.perf_counter()
            pool.map(_oracle_job, jobs, chunksize=1)
            dt = time.perf_counter() - t0
        out["pool"] = {"value": sum(len(t) for t in texts_b) / dt / 1e6, "unit": UNIT, "cores": procs,
                       "kind": "oracle", "seconds": dt,
                       "sample": "the whole batch, one session per task, a process pool over all host cores"}
    return out


def run_reference(args):
    """The oracle on the host cores: each step encodes a bounded sample."""
    from oracle.vocab import Vocab
    cfg = CONFIGS[args.config]
    texts = cfg["texts"]()
    texts_b = [t.encode() for t in texts]
    vocabs = {v: Vocab.load_merges(os.path.join(VOCABS, v + ".merges")) for v, _ in cfg["runs"]}
    from oracle.encode import encode
    samples = reference_samples(args.config, texts, args.warmup + args.steps)
    times, nbytes, nchars = [], 0, 0
    for step, (data, vname, pat) in enumerate(samples):
        t0 = time.perf_counter()
        encode(data, vocabs[vname], pat)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            nbytes += len(data)
            nchars += len(data.decode("utf-8"))
    tot_t = sum(times)
    value = nbytes / tot_t / 1e6
    sample = ("the whole 16 KiB text per step" if args.config == "C1" else
              "a 40,000-character window of the workload per step" +
              (" (the batch's sessions in turn)" if cfg["batch"] else "") +
              (" (patterns alternating)" if len(cfg["runs"]) > 1 else ""))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": config_line(args.config, texts_b, sum(len(t) for t in texts)),
        "ms_per_1m_chars": tot_t * 1e3 * 1e6 / nchars,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample + ", single-threaded Python", **host_cpu()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --- the CUDA path -------------------------------------------------------------

class Run:
    """One tokenizer and its device-resident inputs and outputs."""

    def __init__(self, torch, pkg, vocab_name, pattern, texts_b, batch):
        import numpy as np
        self.tok = pkg.Tokenizer.from_merges_file(os.path.join(VOCABS, vocab_name + ".merges"), pattern)
        self.batch = batch
        self.texts_b = texts_b
        blob = b"".join(texts_b)
        self.n = len(blob)
        self.d_text = torch.frombuffer(bytearray(blob), dtype=torch.uint8).cuda()
        self.d_ids = torch.empty(max(self.n, 1), dtype=torch.int32, device="cuda")
        self.d_st = torch.zeros(4, dtype=torch.int64, device="cuda")
        if batch:
            starts = np.cumsum([0] + [len(t) for t in texts_b]).astype(np.int64)
            self.d_items = torch.from_numpy(starts).cuda()
            self.d_item_off = torch.zeros(len(texts_b) + 1, dtype=torch.int64, device="cuda")
        # pinned host copies for the end-to-end leg
        self.h_texts = [torch.frombuffer(bytearray(t), dtype=torch.uint8).pin_memory() for t in texts_b]
        self.h_ids = torch.empty(max(self.n, 1), dtype=torch.int32).pin_memory()
        self.h_item_off = (ctypes.c_uint64 * (len(texts_b) + 1))()
        self.n_ids = None

    def device_step(self, stream):
        t = self.tok
        if self.batch:
            t.encode_batch_device(self.d_text.data_ptr(), self.n, self.d_items.data_ptr(), len(self.texts_b),
                                  self.d_ids.data_ptr(), self.n, self.d_item_off.data_ptr(), self.d_st.data_ptr(),
                                  stream)
        else:
            t.encode_device(self.d_text.data_ptr(), self.n, self.d_ids.data_ptr(), self.n, self.d_st.data_ptr(),
                            stream)

    def host_step(self):
        """The host entry point from pinned input into pinned output; returns
        the number of ids."""
        L, h = self.tok._L, self.tok._h
        U8P = ctypes.POINTER(ctypes.c_uint8)
        iptr = ctypes.cast(self.h_ids.data_ptr(), ctypes.POINTER(ctypes.c_int32))
        if self.batch:
            k = len(self.texts_b)
            ptrs = (U8P * k)(*[ctypes.cast(x.data_ptr(), U8P) for x in self.h_texts])
            lens = (ctypes.c_uint64 * k)(*[len(x) for x in self.texts_b])
            rc = L.tok_encode_batch(h, ptrs, lens, k, iptr, self.n, self.h_item_off)
            nout = self.h_item_off[k]
        else:
            cnt = ctypes.c_uint64()
            rc = L.tok_encode(h, ctypes.cast(self.h_texts[0].data_ptr(), U8P), self.n, iptr, self.n,
                              ctypes.byref(cnt))
            nout = cnt.value
        assert rc == 0, "host encode failed: %d" % rc
        return nout


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="C3", choices=sorted(CONFIGS))
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return

    import numpy as np
    import torch
    import exact_bpe_tokenization_utf_gb300 as pkg
    from exact_bpe_tokenization_utf_gb300 import _build
    from exact_bpe_tokenization_utf_gb300.shard import assign_items

    cfg = CONFIGS[args.config]
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    _build.build()
    texts = cfg["texts"]()
    texts_b = [t.encode() for t in texts]
    n_chars_all = sum(len(t) for t in texts)
    sharded = cfg["batch"] and world > 1
    if sharded:
        mine = assign_items([len(t) for t in texts_b], world)[rank]
        my_texts = [texts_b[i] for i in mine]
        job_bytes = sum(len(t) for t in texts_b)
    else:
        my_texts = texts_b
        job_bytes = world * sum(len(t) for t in texts_b) * len(cfg["runs"])
    runs = [Run(torch, pkg, vname, pat, my_texts, cfg["batch"]) for vname, pat in cfg["runs"]]
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def step():
        for r in runs:
            r.device_step(sp)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    for r in runs:
        st = r.d_st.cpu().tolist()
        assert st[0] == 0, "encode failed with status %s" % st
        r.n_ids = st[1]

    def timed(k_steps, do_flush):
        ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(k_steps)]
        ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(k_steps)]
        for k in range(k_steps):
            if do_flush:
                flush.zero_()
            ev0[k].record(stream)
            step()
            ev1[k].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in zip(ev0, ev1)]

    def max_over_ranks(x):
        if not dist:
            return x
        t = torch.tensor([x], device="cuda", dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    # timed region: K steps, L2 flushed before each, one pair of events per step
    launches0 = sum(r.tok.launch_count for r in runs)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        step_ms = timed(args.steps, True)
        if dist:
            dist.barrier()
    launches = sum(r.tok.launch_count for r in runs) - launches0
    ms = max_over_ranks(sum(step_ms) / len(step_ms))
    warm_ms = max_over_ranks(statistics.mean(timed(args.steps, False)))

    # per-kernel times: the library's events around each kernel, on the stream
    # the kernels run on, in a separate pass of the same flushed steps (events
    # between the kernels would lengthen the timed steps)
    kern = {}
    kern_steps = min(args.steps, 50)
    for r in runs:
        r.tok.set_timing(True)
    for _ in range(kern_steps):
        flush.zero_()
        step()
        torch.cuda.synchronize()
        per = {}
        for r in runs:
            for nm, t_ms in r.tok.stage_times().items():
                per[nm] = per.get(nm, 0.0) + t_ms
        for nm, t_ms in per.items():
            kern.setdefault(nm, []).append(t_ms)
    for r in runs:
        r.tok.set_timing(False)
        st = r.d_st.cpu().tolist()
        assert st[0] == 0 and st[1] == r.n_ids

    # e2e: host in, host out, from pinned memory, host clock
    e2e_t = []
    for k in range(args.warmup + args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        nouts = [r.host_step() for r in runs]
        t1 = time.perf_counter()
        assert nouts == [r.n_ids for r in runs]
        if k >= args.warmup:
            e2e_t.append(t1 - t0)
    e2e_s = max_over_ranks(sum(e2e_t) / len(e2e_t))
    # the same host calls with the ids returned as Python lists of ints (the
    # list output mode beside the array mode)
    lst_t = []
    for k in range(args.warmup + min(args.steps, 50)):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        lists = [r.h_ids.numpy()[:r.host_step()].tolist() for r in runs]
        t1 = time.perf_counter()
        assert [len(x) for x in lists] == [r.n_ids for r in runs]
        if k >= args.warmup:
            lst_t.append(t1 - t0)
    lst_s = max_over_ranks(sum(lst_t) / len(lst_t))
    ids_ok = all(bool(np.array_equal(r.h_ids.numpy()[:r.n_ids], r.d_ids[:r.n_ids].cpu().numpy())) for r in runs)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    peak, peak_kind = _peaks()
    n_ids = sum(r.n_ids for r in runs)
    my_bytes = sum(r.n for r in runs)
    item_bytes = sum(16 * (len(r.texts_b) + 1) for r in runs if r.batch)
    alg_bytes = my_bytes + 4 * n_ids + item_bytes
    kern_avg = {k: sum(v) / len(v) for k, v in kern.items()}
    top = max(kern_avg, key=kern_avg.get)
    top_ms = kern_avg[top]
    achieved = alg_bytes / (top_ms * 1e-3) / 1e9
    value = job_bytes / (ms * 1e-3) / 1e6
    config = config_line(args.config, texts_b, n_chars_all)
    config["parallelism"] = ("batch sharded over %d ranks" % world if sharded else
                             "%d replicas" % world if world > 1 else "single GPU")
    chars_per_step = n_chars_all * len(cfg["runs"])
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "strong" if sharded else "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": config,
        "ms_per_1m_chars": ms * 1e6 / (n_chars_all if sharded else world * chars_per_step),
        "tokens_per_step": n_ids,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": _traffic(args.config, top), "kernel": top,
                     "note": "algorithmic bytes per step = input bytes + 4 * ids%s = %d, over the dominant "
                             "kernel's time per step; peak = %s copy bandwidth" % (
                                 " + item offsets" if item_bytes else "", alg_bytes, peak_kind)},
        "step_roofline_frac": (alg_bytes / (ms * 1e-3) / 1e9) / peak,
        "kernels_ms": kern_avg,
        "kernels_timing": "library events around each kernel on its stream, %d further flushed steps" % kern_steps,
        "warm_l2": {"ms_per_step": warm_ms, "value": job_bytes / (warm_ms * 1e-3) / 1e6, "unit": UNIT,
                    "note": "the same steps without the L2 flush: vocabulary tables and text L2-resident"},
        "e2e": {"value": job_bytes / e2e_s / 1e6, "unit": UNIT, "h2d_bytes_per_step": my_bytes,
                "d2h_bytes_per_step": 4 * n_ids + 32 * len(runs), "ms_per_step": e2e_s * 1e3},
        "e2e_python_list": {"value": job_bytes / lst_s / 1e6, "unit": UNIT, "ms_per_step": lst_s * 1e3,
                            "note": "the e2e call with the ids converted to Python lists of ints"},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "ids_match_host_path": ids_ok,
    }
    if world == 1 and not args.no_cpu_baseline:
        from oracle.vocab import Vocab
        vocabs = {v: Vocab.load_merges(os.path.join(VOCABS, v + ".merges")) for v, _ in cfg["runs"]}
        line["cpu_baseline"] = cpu_baseline(args.config, texts_b, vocabs)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
