"""Benchmark: fresh-session exact BPE encode of a 1,000,000-character
synthetic agent session (cl100k-style pattern, 256 + 100,000 merges).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one full encode (UTF-8 decode, pre-tokenization, BPE, id scatter)
of the resident input through tok_encode_device.  Between timed steps a
256 MiB buffer is written to flush L2 (the input is smaller than L2).  Each
step is timed with CUDA events on the stream the kernels run on; per-kernel
times come from the library's own events around each kernel.  `e2e` times
tok_encode (host in, host out) from pinned host memory with the host clock.

With N > 1 (torchrun) every rank encodes its own copy of the session (the
path does not shard a single text; replicas, weak scaling) and rank 0 prints
one JSON line with the max time over ranks.

--impl reference times the oracle (plain Python, one core) on a bounded
sample of the same session per step; rank 0 only.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MB/s and ms per 1M chars, IDs bit-exact vs oracle; % of HBM roofline"
UNIT = "MB/s"
VOCAB = os.path.join(ROOT, "data", "vocabs", "cl100k_session_100k.merges")
N_CHARS = 1_000_000
SEED = 1003
WORKLOAD = ("cl100k-style pattern, 256 + 100,000 merges trained on a seeded 64 MiB session corpus; "
            "one 1,000,000-character synthetic agentic session (fresh-session init)")


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if
    the kernel sources have not changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("sources_sha256") != _sources_hash():
        return None
    e = d.get("kernels", {}).get(kernel)
    if not e:
        return None
    return e.get("bytes_per_full_launch")


def _sources_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_bpe_tokenization_utf_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".inc")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode() + fh.read())
    return h.hexdigest()


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


def run_reference(args):
    """The oracle on the host cores: each step encodes a bounded sample."""
    import textgen
    from oracle.encode import encode
    from oracle.pretokenize import PATTERN_CL100K
    from oracle.vocab import Vocab

    v = Vocab.load_merges(VOCAB)
    text = textgen.agentic_session(N_CHARS, SEED)
    sample_chars = 40_000
    times, nbytes = [], []
    for step in range(args.warmup + args.steps):
        a = (step * 97_003) % (N_CHARS - sample_chars)
        piece = text[a:a + sample_chars].encode()
        t0 = time.perf_counter()
        encode(piece, v, PATTERN_CL100K)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            nbytes.append(len(piece))
    tot_t, tot_b = sum(times), sum(nbytes)
    value = tot_b / tot_t / 1e6
    ms_per_1m = (tot_t / len(times)) * 1e3 * 1e6 / sample_chars
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": "%d-character windows of the session per step" % sample_chars},
        "ms_per_1m_chars": ms_per_1m,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "%d-character windows of the 1M-character session, one per step" % sample_chars},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(text_bytes):
    """The oracle, as it stands, on one host core over a bounded sample."""
    from oracle.encode import encode
    from oracle.pretokenize import PATTERN_CL100K
    from oracle.vocab import Vocab
    v = Vocab.load_merges(VOCAB)
    sample = text_bytes
    t0 = time.perf_counter()
    encode(sample, v, PATTERN_CL100K)
    dt = time.perf_counter() - t0
    return {"value": len(sample) / dt / 1e6, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "the whole session (%d bytes), single-threaded Python" % len(sample),
            "seconds": dt}


def main():
    ap = argparse.ArgumentParser()
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
    import textgen
    from exact_bpe_tokenization_utf_gb300 import PATTERN_CL100K, Tokenizer
    from exact_bpe_tokenization_utf_gb300 import _build

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    _build.build()
    tok = Tokenizer.from_merges_file(VOCAB, PATTERN_CL100K)
    text = textgen.agentic_session(N_CHARS, SEED)
    data = text.encode()
    n = len(data)
    stream = torch.cuda.current_stream()
    d_text = torch.frombuffer(bytearray(data), dtype=torch.uint8).cuda()
    d_ids = torch.empty(n, dtype=torch.int32, device="cuda")
    d_st = torch.zeros(4, dtype=torch.int64, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def step():
        tok.encode_device(d_text.data_ptr(), n, d_ids.data_ptr(), n, d_st.data_ptr(), stream.cuda_stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    st = d_st.cpu().tolist()
    assert st[0] == 0, "encode failed with status %s" % st
    n_ids = st[1]

    # timed region: K steps, L2 flushed before each, one pair of events per step
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    launches0 = tok.launch_count
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for k in range(args.steps):
            flush.zero_()
            ev0[k].record(stream)
            step()
            ev1[k].record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
    launches = tok.launch_count - launches0
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]

    # per-kernel times: the library's events around each kernel, on the stream
    # the kernels run on, in a separate pass of the same steps (events between
    # the kernels would lengthen the timed steps)
    kern = {}
    kern_steps = min(args.steps, 50)
    tok.set_timing(True)
    for k in range(kern_steps):
        flush.zero_()
        step()
        torch.cuda.synchronize()
        for nm, ms in tok.stage_times().items():
            kern.setdefault(nm, []).append(ms)
    tok.set_timing(False)
    ms = sum(step_ms) / len(step_ms)
    if dist:
        t = torch.tensor([ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    st = d_st.cpu().tolist()
    assert st[0] == 0 and st[1] == n_ids

    # e2e: host in, host out, from pinned memory, host clock
    h_text = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    h_text.numpy()[:] = np.frombuffer(data, dtype=np.uint8)
    h_ids = torch.empty(n, dtype=torch.int32, pin_memory=True)
    import ctypes
    L = tok._L
    nout = ctypes.c_uint64()
    tptr = ctypes.cast(h_text.data_ptr(), ctypes.POINTER(ctypes.c_uint8))
    iptr = ctypes.cast(h_ids.data_ptr(), ctypes.POINTER(ctypes.c_int32))
    e2e_t = []
    for k in range(args.warmup + args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        rc = L.tok_encode(tok._h, tptr, n, iptr, n, ctypes.byref(nout))
        t1 = time.perf_counter()
        assert rc == 0 and nout.value == n_ids
        if k >= args.warmup:
            e2e_t.append(t1 - t0)
    e2e_s = sum(e2e_t) / len(e2e_t)
    if dist:
        t = torch.tensor([e2e_s], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_s = float(t.item())
    ids_ok = bool(np.array_equal(h_ids.numpy()[:n_ids], d_ids[:n_ids].cpu().numpy()))

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    peak, peak_kind = _peaks()
    alg_bytes = n + 4 * n_ids
    kern_avg = {k: sum(v) / len(v) for k, v in kern.items()}
    top = max(kern_avg, key=kern_avg.get)
    top_ms = kern_avg[top]
    achieved = alg_bytes / (top_ms * 1e-3) / 1e9
    value = world * n / (ms * 1e-3) / 1e6
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "bytes": n, "chars": N_CHARS, "tokens": n_ids,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "flushed before every timed step (256 MiB write)"},
        "ms_per_1m_chars": ms * 1e6 / N_CHARS,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": _traffic(top), "kernel": top,
                     "note": "algorithmic bytes = input bytes + 4 * ids = %d per launch; peak %s" % (
                         alg_bytes, peak_kind)},
        "step_roofline_frac": (alg_bytes / (ms * 1e-3) / 1e9) / peak,
        "kernels_ms": kern_avg,
        "kernels_timing": "library events around each kernel on its stream, %d further flushed steps" % kern_steps,
        "e2e": {"value": world * n / e2e_s / 1e6, "unit": UNIT, "h2d_bytes_per_step": n,
                "d2h_bytes_per_step": 4 * n_ids + 64, "ms_per_step": e2e_s * 1e3},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "ids_match_host_path": ids_ok,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(data)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
