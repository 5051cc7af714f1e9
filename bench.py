"""Benchmark of one absorbed-MLA decode step on a GB300 (prints ONE JSON line on rank 0).

A step is the whole hot path over one batch: mla_kv_append of each sequence's
new row, then mla_decode (planner, query absorption, split-KV flash decode over
the paged latent cache, log-sum-exp combine + W_UV up-projection).

Default workload: DeepSeek-V3 shapes, B = 64 sequences of 4096 tokens, bf16
cache (n_h = 128, d_c = 512, d_rope = 64).  Metric: latent-KV GB/s, i.e. the
decode-step cache read B * s_ctx * (d_c + d_rope) * e bytes ("G5 MLA KV
访存建模设计规格" eq. gmkv-read) divided by the step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

--impl reference times the CPU fp64 oracle (the reference arm of this method)
on the host cores on a bounded sample of the same workload.
Under torchrun each rank runs an independent replica (the path has no
cross-sequence exchange), value = all ranks' bytes / max-over-ranks time.
"""
from __future__ import annotations

import os
import sys

# The CPU oracle legs use every host core through BLAS; fix the thread count
# before numpy is imported so the reported core count is the one used.
_CORES = os.cpu_count() or 1
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "absorbed-MLA decode µs/step, latent-KV GB/s and % of roofline at B×s_ctx"
DECODE_SOURCES = ["mla_absorbed_latent_decode_gb300/csrc/decode_tc.cu"]
PREFILL_SOURCES = ["mla_absorbed_latent_decode_gb300/csrc/prefill.cu"]


def parse():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="v3_b64_s4096_bf16")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--naive-ab", action="store_true",
                    help="also time the standard-mode decode over the expanded per-head cache (bf16 cache only)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU seconds of the oracle baseline sample")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


LAYER = "v2lite_layer"      # the V2-Lite layer step with its projections on the GPU


PREFILL = "v3_prefill_b2_s4096"   # whole-prompt prefill, MHA mode (a compute-bound second workload)


def workload(name):
    from mla_absorbed_latent_decode_gb300 import workloads as W
    if name == PREFILL:
        return W.v3_prefill()
    if name == LAYER:
        # x -> W_Q, W_DKV on the device (mla_project, mla_kv_project_append), then the decode;
        # the workload's rows and query are placeholders until the CPU leg projects them
        inp = W.v2lite_single_step_inputs(seed=0)
        rows = np.zeros((inp["tokens"], W.D_C + W.D_ROPE), np.uint16)
        q = np.zeros((inp["n_h"], W.D_NOPE + W.D_ROPE), np.uint16)
        wl = W.v2lite_single_step(rows, q, inp["w_uk"], inp["w_uv"], n_h=inp["n_h"])
        wl.name = LAYER
        wl.extra["layer"] = inp
        return wl
    if name in W.EXTRA:
        return W.EXTRA[name]()
    if name not in W.NAMED:
        raise SystemExit(f"unknown workload {name}; choose from {sorted(W.NAMED) + sorted(W.EXTRA) + [LAYER, PREFILL]}")
    return W.NAMED[name]()


def algorithmic(wl):
    """Bytes and FLOPs of one decode step (cache + W_UK + W_UV bytes; QK^T, P.c_kv, absorb, W_UV flops)."""
    tokens = wl.total_tokens
    cache = tokens * cache_bytes_per_token(wl)
    weights = 2 * wl.n_h * 128 * 512 * 2
    flops = 2 * wl.n_h * tokens * (576 + 512) + 4 * wl.B * wl.n_h * 128 * 512
    if "layer" in wl.extra:                            # + W_Q and W_DKV for the step's token
        proj = (wl.n_h * (wl.d_nope + wl.d_rope) + wl.d_c + wl.d_rope) * wl.extra["layer"]["x"].shape[1]
        weights += 2 * proj
        flops += 2 * wl.B * proj
    return cache, weights, flops


def prefill_flops(wl):
    """FLOPs of one prefill step: the per-head expansion of every cached row (W_UK and W_UV,
    2 n_h (d_nope + d_v) d_c per row) and the causal attention (2 n_h (d_nope + d_rope + d_v)
    per visible query-key pair); returns (expansion, attention)."""
    p = wl.extra["prefill"]
    rows = int(np.sum(wl.ctx_len.astype(np.int64)))
    expand = 2 * wl.n_h * (wl.d_nope + wl.d_v) * wl.d_c * rows
    pairs = 0
    for L, n in zip(wl.ctx_len.astype(np.int64), p["q_len"].astype(np.int64)):
        pairs += n * (L - n) + n * (n + 1) // 2          # query i sees L - n + i + 1 keys
    attn = 2 * wl.n_h * (wl.d_nope + wl.d_rope + wl.d_v) * pairs
    return expand, attn


def cache_bytes_per_token(wl):
    from mla_absorbed_latent_decode_gb300 import workloads as W
    return W.ROW_BYTES[wl.cache_dtype]          # 1152 bf16, 576 e4m3, 656 per-block e4m3 (+ scales, bf16 RoPE)


def cache_name(wl):
    return {1: "bf16", 2: "fp8_e4m3", 3: "fp8_e4m3_block"}[wl.cache_dtype]


def ranks_max(values, device, world):
    """Each value's maximum over the ranks: the slowest rank sets a whole-job time."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_rate(world, units_per_rank, ms):
    """Whole-job throughput per second: every rank processes `units_per_rank` (replicas, weak
    scaling) and the job takes the slowest rank's `ms`."""
    return world * units_per_rank / (ms * 1e-3)


# ------------------------------------------------------------------ CPU oracle leg

def oracle_sample(wl, seconds):
    """Time the oracle's absorbed decode on the first sequences of the workload until
    about `seconds` of CPU work; return (GB/s of latent cache processed, description)."""
    from oracle import mla_ref
    from oracle import e4m3
    if "layer" in wl.extra and "projected" not in wl.extra:
        inp = wl.extra["layer"]
        c, kr, qq = mla_ref.project_inputs(mla_ref.bf16_to_f64(inp["x"]), mla_ref.bf16_to_f64(inp["w_dkv"]),
                                           mla_ref.bf16_to_f64(inp["w_q"]), inp["n_h"], wl.d_c)
        wl.rows = mla_ref.bf16_round(np.concatenate([c, kr], axis=1).astype(np.float32))
        wl.q = mla_ref.bf16_round(qq[-1].astype(np.float32)).reshape(1, inp["n_h"], -1)
        wl.extra["projected"] = True
    starts = np.concatenate([[0], np.cumsum(wl.ctx_len.astype(np.int64))])
    q = mla_ref.bf16_to_f64(wl.q)
    w_uk = mla_ref.bf16_to_f64(wl.w_uk)
    w_uv = mla_ref.bf16_to_f64(wl.w_uv)
    scale = mla_ref.default_scale(wl.d_nope, wl.d_rope)
    done_tokens, elapsed, nseq = 0, 0.0, 0
    cached = wl.extra.setdefault("oracle_values", {})
    for i in range(100 * wl.B):                       # cycles through the batch until `seconds` is reached
        b = i % wl.B
        a, z = starts[b], starts[b + 1]
        if b not in cached:                 # the oracle's own cache contents (prefill, untimed)
            if wl.cache_dtype == 3:
                st = mla_ref.stored_row_fp8_block(wl.rows[a:z], wl.row_pos[a:z], wl.d_c, wl.rope_base)
                cached[b] = mla_ref.fp8_block_values(st, wl.d_c)
            elif wl.cache_dtype == 2:
                st = mla_ref.stored_row_e4m3(wl.rows[a:z], wl.row_pos[a:z], wl.d_c, wl.rope_base,
                                             np.float32(wl.fp8_scale))
                cached[b] = e4m3.decode(st) * float(np.float32(wl.fp8_scale))
            else:
                cached[b] = mla_ref.bf16_to_f64(mla_ref.stored_row_bf16(wl.rows[a:z], wl.row_pos[a:z], wl.d_c,
                                                                        wl.rope_base))
        vals = cached[b]
        t0 = time.perf_counter()
        mla_ref.absorbed_decode(q[b], vals[:, :wl.d_c], vals[:, wl.d_c:], w_uk, w_uv, int(wl.ctx_len[b]) - 1,
                                scale, wl.rope_base)
        elapsed += time.perf_counter() - t0
        done_tokens += int(z - a)
        nseq += 1
        if elapsed >= seconds:
            break
    gbps = done_tokens * cache_bytes_per_token(wl) / elapsed / 1e9
    return gbps, elapsed, (f"{nseq} sequence decodes over the first {min(nseq, wl.B)} of {wl.B} sequences "
                           f"({done_tokens} tokens), fp64 absorbed path, {elapsed:.1f} s")


def arithmetic_note(wl):
    """What the decode computes in, for the JSON line's config."""
    if cache_name(wl) == "fp8_e4m3":
        ops = ("e4m3 MMA operands (the cached codes as stored, the absorbed query quantised per head and "
               "half, P in e4m3; the RoPE part in bf16)")
    elif cache_name(wl) == "fp8_e4m3_block":
        ops = "bf16 MMA operands (the per-block e4m3 cache decoded to bf16 in shared memory)"
    else:
        ops = "bf16 MMA operands"
    return ops + ", fp32 accumulation and softmax, fp16 partial scores between the CTA pair"


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return int(os.environ.get("OPENBLAS_NUM_THREADS", _CORES))


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    wl = workload(args.workload)
    per_step = max(0.5, min(3.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(wl, per_step)
    vals, secs = [], []
    for _ in range(args.steps):
        g, el, desc = oracle_sample(wl, per_step)
        vals.append(g)
        secs.append(el)
    v = statistics.mean(vals)
    us_equiv = wl.total_tokens * cache_bytes_per_token(wl) / (v * 1e9) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s (latent KV)",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(us_equiv / 1000.0, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "s_ctx": wl.max_ctx, "n_h": wl.n_h, "d_c": wl.d_c,
                   "d_rope": wl.d_rope, "cache": cache_name(wl), "total_tokens": wl.total_tokens,
                   "parallelism": "replicas x1 (rank 0 only)",
                   "note": "ms_per_step extrapolated from the sampled throughput to the whole batch"},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s (latent KV)", "cores": blas_threads(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(v, 4), "unit": "GB/s (latent KV)", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU leg

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc, self.gpu = None, gpu_index
        out_dir = os.environ.get("MLA_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"mla_bench_clocks_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sms, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sms)}


def source_hash(sources=DECODE_SOURCES):
    h = hashlib.sha256()
    for rel in sources:
        p = os.path.join(ROOT, rel)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()


def ncu_traffic(wl, summary="decode_traffic.json", sources=DECODE_SOURCES):
    """Per-launch DRAM bytes of a kernel from a committed ncu summary, if it was taken on the
    current source of that kernel for this workload; else None."""
    p = os.path.join(ROOT, "profiles", summary)
    try:
        d = json.load(open(p))
    except Exception:
        return None
    if d.get("source_sha256") != source_hash(sources) or d.get("workload") != wl.name:
        return None
    return d.get("bytes_per_launch")


def pipelined_e2e(stream, dev, h_pack, d_packs, outs, h_outs, slot_step, steps, warmup):
    """End-to-end steps as a serving loop runs them: two slots of device inputs and outputs; the
    host-to-device copy of step i + 1 and the read-back of step i - 1 run on their own streams
    while step i computes.  `slot_step(k)` issues the step on slot k's buffers (the public API
    calls) on the current stream; each slot's step is captured once in a CUDA graph and replayed.
    The timed region starts before the first copy in and ends when the last result is on the
    host.  Returns ms per step."""
    import torch
    side = torch.cuda.Stream(device=dev)
    graphs = []
    for k in range(2):
        g = torch.cuda.CUDAGraph()
        side.wait_stream(stream)
        with torch.cuda.graph(g, stream=side):
            slot_step(k)
        graphs.append(g)
    stream.wait_stream(side)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    read = [torch.cuda.Event(), torch.cuda.Event()]

    def run(k_steps, start=None):
        if start is not None:
            s_in.wait_event(start)
        for i in range(k_steps):
            k = i % 2
            if i >= 2:
                s_in.wait_event(done[k])             # step i - 2 has read this slot's inputs
            with torch.cuda.stream(s_in):
                d_packs[k].copy_(h_pack, non_blocking=True)
            in_ready[k].record(s_in)
            stream.wait_event(in_ready[k])
            if i >= 2:
                stream.wait_event(read[k])           # step i - 2's result has left this slot
            graphs[k].replay()
            done[k].record(stream)
            s_out.wait_event(done[k])
            with torch.cuda.stream(s_out):
                h_outs[k].copy_(outs[k].view(torch.int16), non_blocking=True)
            read[k].record(s_out)
        stream.wait_event(read[(k_steps - 1) % 2])

    run(max(2, warmup))
    torch.cuda.synchronize()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    run(steps, start=p0)
    p1.record(stream)
    p1.synchronize()
    return p0.elapsed_time(p1) / steps


E2E_MODE = ("pipelined: the copies of steps i + 1 (in) and i - 1 (out) overlap step i's compute; each of the "
            "two buffer slots' steps (the same public calls) replayed from a CUDA graph captured once")


def run_ours(args):
    import torch
    import torch.distributed as dist

    from mla_absorbed_latent_decode_gb300 import binding as B
    from mla_absorbed_latent_decode_gb300.runner import DecodeSession, bf16_tensor

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    wl = workload(args.workload)
    sess = DecodeSession(wl, device=str(dev))
    layer = "layer" in wl.extra
    if layer:
        inp = wl.extra["layer"]
        T, qw = inp["tokens"], wl.n_h * (wl.d_nope + wl.d_rope)
        x_all = bf16_tensor(inp["x"], dev)
        w_q, w_dkv = bf16_tensor(inp["w_q"], dev), bf16_tensor(inp["w_dkv"], dev)
        lseq = torch.zeros(T, dtype=torch.int32, device=dev)
        lpos = torch.arange(T, dtype=torch.int32, device=dev)
        sess.mla.kv_project_append(x_all[:T - 1], w_dkv, lseq[:T - 1], lpos[:T - 1], sess.block_table, sess.cache,
                                   wl.num_pages)                              # the 25-token prefill
        x_new = x_all[T - 1:]
        q_new = torch.empty((1, qw), dtype=torch.bfloat16, device=dev)
    else:
        sess.prefill()
        rows, seq, pos = sess.step_inputs()
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    flush_rd = torch.ones_like(flush)

    def flush_l2():
        """Cold L2 for the next step: write a buffer twice the L2 size, then read another one
        of that size, so that L2 ends up holding clean lines only and no write-back of the
        flush's own dirty lines lands inside the next timed step."""
        flush.zero_()
        flush_rd.view(torch.int32).amax()
    sess.mla.set_option(B.MLA_OPT_PROFILE, 1)

    def step():
        if layer:                     # the new token's q and cache row projected on the device
            sess.mla.project(x_new, w_q, q_new)
            sess.mla.kv_project_append(x_new, w_dkv, lseq[T - 1:], lpos[T - 1:], sess.block_table, sess.cache,
                                       wl.num_pages)
            sess.decode(q=q_new.view(1, wl.n_h, -1))
        else:
            sess.append_step(rows, seq, pos)
            sess.decode()

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    if sess.status() != 0:
        raise SystemExit("device check word set during warm-up")

    def timed_pass(profile, flush=True):
        """K steps, each bracketed by CUDA events on the stream (L2 flushed between steps,
        outside the events, unless flush=False).  With profile=True the library also records
        events around each of its kernels (which serialises them); returns per-step ms and
        per-kernel ms."""
        sess.mla.set_option(B.MLA_OPT_PROFILE, 1 if profile else 0)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        kms = []
        for i in range(args.steps):
            if flush:
                flush_l2()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
            if profile:
                kms.append(sess.mla.profile_read())      # syncs this step's events (between steps)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in zip(starts, ends)], kms

    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    step_ms, _ = timed_pass(profile=False)      # the headline: the step as a user runs it
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    _, kernel_ms = timed_pass(profile=True)    # per-kernel device times for the roofline
    torch.cuda.synchronize()
    warm_ms, _ = timed_pass(profile=False, flush=False)   # reported beside: no flush between steps
    torch.cuda.synchronize()
    # reported beside: the same step captured once in a CUDA graph and replayed (every per-step
    # decision is made on the device, so the captured launches serve every step)
    sess.mla.set_option(B.MLA_OPT_PROFILE, 0)
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step()
    graph_ms = []
    for _ in range(max(1, args.warmup)):
        flush_l2()
        graph.replay()
    for _ in range(args.steps):
        flush_l2()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        z.record(stream)
        z.synchronize()
        graph_ms.append(a.elapsed_time(z))
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    ms = statistics.mean(step_ms)
    ms_median = statistics.median(step_ms)
    warm = statistics.mean(warm_ms)
    if sess.status() != 0:
        raise SystemExit("device check word set during the timed steps")

    # end to end through the public API with host buffers: H2D of the step's inputs,
    # append + decode, D2H of the result, every step
    # the step's inputs travel in one pinned host buffer and one copy (a copy has a fixed cost
    # of several microseconds; five small ones cost more than the 3 MB of queries); each input
    # is a 256-byte aligned segment of the packed buffer
    last = wl.last_row_index()
    if layer:                         # the step's input is the new token's hidden state
        parts = [("x", inp["x"][T - 1:].view(np.int16)), ("seq", np.zeros(1, np.int32)),
                 ("pos", np.array([T - 1], np.int32)), ("ctx", wl.ctx_len.astype(np.int32))]
    else:
        parts = [("rows", wl.rows[last].view(np.int16)), ("seq", wl.row_seq[last].astype(np.int32)),
                 ("pos", wl.row_pos[last].astype(np.int32)), ("q", wl.q.view(np.int16)),
                 ("ctx", wl.ctx_len.astype(np.int32))]
    offs, total = {}, 0
    for name, a in parts:
        offs[name] = total
        total += (a.nbytes + 255) // 256 * 256
    h_pack = torch.empty(total, dtype=torch.uint8).pin_memory()
    d_pack = torch.empty(total, dtype=torch.uint8, device=dev)
    views = {}
    for name, a in parts:
        flat = np.ascontiguousarray(a).reshape(-1)
        h_pack[offs[name]:offs[name] + flat.nbytes].copy_(torch.from_numpy(flat.view(np.uint8)))
        dt = torch.int16 if flat.dtype == np.int16 else torch.int32
        views[name] = d_pack[offs[name]:offs[name] + flat.nbytes].view(dt).view(a.shape)
    h_out = torch.empty((wl.B, wl.n_h, wl.d_v), dtype=torch.int16).pin_memory()
    h2d = sum(a.nbytes for _, a in parts)
    d2h = h_out.numel() * h_out.element_size()
    sess.mla.set_option(B.MLA_OPT_PROFILE, 0)

    def compute(v, out):
        """The step through the public API on the current stream, inputs in the views `v`."""
        if layer:
            xv = v["x"].view(torch.bfloat16)
            sess.mla.project(xv, w_q, q_new)
            sess.mla.kv_project_append(xv, w_dkv, v["seq"], v["pos"], sess.block_table, sess.cache, wl.num_pages)
            sess.mla.decode(q_new.view(1, wl.n_h, -1), v["ctx"], wl.max_ctx, sess.block_table, sess.cache,
                            wl.num_pages, sess.workspace, out)
        else:
            sess.mla.kv_append(v["rows"].view(torch.bfloat16), v["seq"], v["pos"], sess.block_table, sess.cache,
                               wl.num_pages)
            sess.mla.decode(v["q"].view(torch.bfloat16), v["ctx"], wl.max_ctx, sess.block_table, sess.cache,
                            wl.num_pages, sess.workspace, out)

    def e2e_step():
        d_pack.copy_(h_pack, non_blocking=True)
        compute(views, sess.out)
        h_out.copy_(sess.out.view(torch.int16), non_blocking=True)

    for _ in range(max(1, args.warmup)):
        flush_l2()
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for i in range(args.steps):
        flush_l2()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        e2e_step()
        s1.record(stream)
        s1.synchronize()
        e2e_ms.append(s0.elapsed_time(s1))
    e2e_serial = statistics.mean(e2e_ms)

    # the same steps as a serving loop runs them (the inputs, the 288 MiB cache read per step,
    # exceed L2)
    d_packs = [d_pack, torch.empty_like(d_pack)]
    views_k = [views, {}]
    for name, a in parts:
        n = np.ascontiguousarray(a).nbytes
        dt = torch.int16 if np.asarray(a).dtype == np.int16 else torch.int32
        views_k[1][name] = d_packs[1][offs[name]:offs[name] + n].view(dt).view(a.shape)
    outs = [sess.out, torch.empty_like(sess.out)]
    h_outs = [h_out, torch.empty_like(h_out).pin_memory()]
    e2e = pipelined_e2e(stream, dev, h_pack, d_packs, outs, h_outs, lambda k: compute(views_k[k], outs[k]),
                        args.steps, args.warmup)
    naive = naive_ab(args, wl, sess, flush_l2, stream) if args.naive_ab and not layer else None

    ms, e2e, warm, graph_mean = ranks_max([ms, e2e, warm, statistics.mean(graph_ms)], dev, world)

    cache_b, weight_b, flops = algorithmic(wl)
    hbm, tc_burst, tc_sust, peak_kind = peaks()
    value = job_rate(world, cache_b, ms) / 1e9
    e2e_value = job_rate(world, cache_b, e2e) / 1e9
    roof_us = max((cache_b + weight_b) / (hbm * 1e9), flops / (tc_burst * 1e12)) * 1e6
    dec_ms = statistics.mean(k.get("mla_decode_splitkv", float("nan")) for k in kernel_ms)
    per_kernel = {k: round(statistics.mean(km[k] for km in kernel_ms) * 1000.0, 2) for k in kernel_ms[0]}
    achieved = cache_b / (dec_ms * 1e-3) / 1e9
    traffic = ncu_traffic(wl)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s (latent KV)", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "us_per_step": round(ms * 1000.0, 2), "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
            "roofline_us": round(roof_us, 2), "roofline_frac_step": round(roof_us / (ms * 1000.0), 4),
            "us_per_step_median": round(ms_median * 1000.0, 2),
            "total_gbs": round(job_rate(world, cache_b + weight_b, ms) / 1e9, 1),
            "warm_l2": {"us_per_step": round(warm * 1000.0, 2),
                        "value": round(job_rate(world, cache_b, warm) / 1e9, 2), "unit": "GB/s (latent KV)",
                        "note": "the same K steps back to back with no flush between them (weights and "
                                "part of the cache may stay in L2); not the headline"},
            "graph_replay": {"us_per_step": round(graph_mean * 1000.0, 2),
                             "value": round(job_rate(world, cache_b, graph_mean) / 1e9, 2),
                             "unit": "GB/s (latent KV)",
                             "note": "the same step captured once in a CUDA graph and replayed, L2 flushed "
                                     "between replays; not the headline"},
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3" if cache_name(wl) == "fp8_e4m3" else "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.B, "s_ctx": wl.max_ctx, "n_h": wl.n_h, "d_c": wl.d_c,
                       "d_rope": wl.d_rope, "cache": cache_name(wl),
                       "total_tokens": wl.total_tokens,
                       "l2": f"flushed between steps outside the timed events: write of {flush.numel() >> 20} MiB, "
                             f"then read of another {flush_rd.numel() >> 20} MiB (L2 left cold and clean); the "
                             f"cache read per step ({wl.total_tokens * cache_bytes_per_token(wl) >> 20} MiB) also exceeds L2",
                       "timing": "value from K steps without per-kernel events; per_kernel_us and roofline "
                                 "from a second K-step pass with per-kernel events (which serialise the kernels)",
                       "arithmetic": arithmetic_note(wl),
                       "parallelism": f"replicas x{world}"},
            "per_kernel_us": per_kernel,
            "roofline": {"bound": "hbm", "kernel": "mla_decode_splitkv", "achieved": round(achieved, 1),
                         "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                         "traffic": traffic, "peak_source": f"{peak_kind} hbm_gbs",
                         "algorithmic_bytes_per_launch": cache_b},
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s (latent KV)", "ms_per_step": round(e2e, 5),
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "mode": E2E_MODE,
                    "l2": (f"not flushed between pipelined steps (a flush would serialise the copies); each step "
                           f"reads {wl.total_tokens * cache_bytes_per_token(wl) >> 20} MiB of cache, more than L2; "
                           f"serial_ms_per_step flushes L2 before every step"),
                    "serial_ms_per_step": round(e2e_serial, 5)},
            "gpu_launches": args.steps * ((2 if layer else 1) + len(kernel_ms[0])),
            "clocks": clock_info,
        }
        if layer:
            line["config"]["projections"] = ("the new token's q = x . W_Q and cache row = x . W_DKV computed on "
                                             "the device (mla_project, mla_kv_project_append) inside the step")
        if naive is not None:
            naive["absorbed_step_us"] = round(ms * 1000.0, 2)
            naive["naive_over_absorbed"] = round(naive["decode_us"] / (ms * 1000.0), 2)
            naive["frac_of_hbm"] = round(naive["gbs"] / hbm, 4)
            line["naive_ab"] = naive
        if world == 1 and not args.no_cpu_baseline:
            g, el, desc = oracle_sample(wl, args.cpu_seconds)
            line["cpu_baseline"] = {"value": round(g, 4), "unit": "GB/s (latent KV)", "cores": blas_threads(),
                                    "kind": "oracle", "sample": desc}
        print(json.dumps(line), flush=True)
    sess.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def naive_ab(args, wl, sess, flush_l2, stream):
    """Standard-mode decode of the same batch: the latent cache expanded once into per-head keys
    [W_UK c ; k_r] and values W_UV c (mla_expand_kv, untimed), then K decode calls over it
    (mla_decode_naive), L2 flushed between calls.  The bytes it must read per call are
    B * s_ctx * n_h * (d_nope + d_rope + d_v) * 2 -- the per-token cache of a standard MHA."""
    import torch
    if wl.cache_dtype != 1:
        return None
    mla = sess.mla
    kvx = torch.empty((wl.num_pages, wl.page_size, wl.n_h, wl.d_nope + wl.d_rope + wl.d_v), dtype=torch.bfloat16,
                      device=sess.cache.device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    mla.expand_kv(sess.cache, wl.num_pages, kvx)
    e1.record(stream)
    ws = torch.empty(mla.decode_naive_workspace_size(wl.B, wl.max_ctx), dtype=torch.uint8, device=kvx.device)
    out = torch.empty_like(sess.out)

    def call():
        mla.decode_naive(sess.q, sess.ctx_len, wl.max_ctx, sess.block_table, kvx, wl.num_pages, ws, out)
    for _ in range(max(3, args.warmup)):
        flush_l2()
        call()
    torch.cuda.synchronize()
    times = []
    for _ in range(args.steps):
        flush_l2()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        call()
        s1.record(stream)
        torch.cuda.synchronize()
        times.append(s0.elapsed_time(s1))
    if sess.status() != 0:
        raise SystemExit("device check word set during the standard-mode decode")
    us = statistics.mean(times) * 1000.0
    xbytes = wl.total_tokens * wl.n_h * (wl.d_nope + wl.d_rope + wl.d_v) * 2
    res = {"decode_us": round(us, 2), "expanded_bytes_per_step": int(xbytes), "gbs": round(xbytes / (us * 1e3), 1),
           "expand_ms_once": round(e0.elapsed_time(e1), 2),
           "note": "standard-mode decode (expanded per-head K/V, no absorption) over the same batch; "
                   "decode call only, L2 flushed between calls"}
    del kvx
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------ prefill workload

def prefill_oracle_sample(wl, seconds):
    """Time the oracle's MHA-mode prefill of sequence 0, one head at a time, until about
    `seconds` of CPU work; return (algorithmic TFLOP/s, seconds, description)."""
    from oracle import mla_ref
    p = wl.extra["prefill"]
    L, n = int(wl.ctx_len[0]), int(p["q_len"][0])
    vals = wl.extra.get("oracle_vals0")
    if vals is None:                                  # the oracle's own cache contents (untimed)
        vals = mla_ref.bf16_to_f64(mla_ref.stored_row_bf16(wl.rows[:L], wl.row_pos[:L], wl.d_c, wl.rope_base))
        wl.extra["oracle_vals0"] = vals
    q = mla_ref.bf16_to_f64(p["q"][:n])
    w_uk, w_uv = mla_ref.bf16_to_f64(wl.w_uk), mla_ref.bf16_to_f64(wl.w_uv)
    scale = mla_ref.default_scale(wl.d_nope, wl.d_rope)
    elapsed, heads = 0.0, 0
    for h in range(wl.n_h):
        t0 = time.perf_counter()
        mla_ref.prefill_naive(q[:, h:h + 1], vals[:, :wl.d_c], vals[:, wl.d_c:], w_uk[h:h + 1], w_uv[h:h + 1], L - n,
                              scale, wl.rope_base)
        elapsed += time.perf_counter() - t0
        heads += 1
        if elapsed >= seconds:
            break
    pairs = n * (L - n) + n * (n + 1) // 2
    flops = heads * (2 * (wl.d_nope + wl.d_v) * wl.d_c * L + 2 * (wl.d_nope + wl.d_rope + wl.d_v) * pairs)
    return flops / elapsed / 1e12, elapsed, (f"{heads} of {wl.n_h} heads of sequence 0 ({L} tokens, {n} queries), "
                                             f"fp64 MHA-mode prefill, {elapsed:.1f} s")


def run_prefill_reference(args, wl):
    per_step = max(0.5, min(3.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        prefill_oracle_sample(wl, per_step)
    vals, desc = [], ""
    for _ in range(args.steps):
        v, _, desc = prefill_oracle_sample(wl, per_step)
        vals.append(v)
    v = statistics.mean(vals)
    fe, fa = prefill_flops(wl)
    line = {
        "impl": "reference", "metric": PREFILL_METRIC, "value": round(v, 6), "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round((fe + fa) / (v * 1e12) * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "s_ctx": wl.max_ctx, "n_h": wl.n_h, "cache": "bf16",
                   "note": "ms_per_step extrapolated from the sampled throughput to the whole batch"},
        "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


PREFILL_METRIC = "MLA prefill (MHA mode, causal) TFLOP/s and % of the bf16 tensor peak"


def run_prefill(args, wl):
    """One step = mla_kv_append of every prompt row + mla_prefill (expansion + attention)."""
    import torch
    import torch.distributed as dist

    from mla_absorbed_latent_decode_gb300 import binding as B
    from mla_absorbed_latent_decode_gb300.runner import DecodeSession, bf16_tensor

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    p = wl.extra["prefill"]
    sess = DecodeSession(wl, device=str(dev))
    rows = bf16_tensor(wl.rows, dev)
    seq = torch.from_numpy(wl.row_seq.astype(np.int32)).to(dev)
    pos = torch.from_numpy(wl.row_pos.astype(np.int32)).to(dev)
    q = bf16_tensor(p["q"], dev)
    q_start = torch.from_numpy(p["q_start"].astype(np.int32)).to(dev)
    q_len = torch.from_numpy(p["q_len"].astype(np.int32)).to(dev)
    max_q = int(p["q_len"].max())
    ws = torch.empty(sess.mla.prefill_workspace_size(wl.B, wl.max_ctx), dtype=torch.uint8, device=dev)
    out = torch.empty((q.shape[0], wl.n_h, wl.d_v), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    flush_rd = torch.ones_like(flush)

    def flush_l2():
        flush.zero_()
        flush_rd.view(torch.int32).amax()

    def step(rows=rows, seq=seq, pos=pos, q=q, q_start=q_start, q_len=q_len, ctx=sess.ctx_len, o=out):
        sess.mla.kv_append(rows, seq, pos, sess.block_table, sess.cache, wl.num_pages)
        sess.mla.prefill(q, q_start, q_len, max_q, ctx, wl.max_ctx, sess.block_table, sess.cache, wl.num_pages,
                         ws, o)

    for _ in range(max(3, args.warmup)):
        flush_l2()
        step()
    torch.cuda.synchronize()
    if sess.status() != 0:
        raise SystemExit("device check word set during warm-up")

    def timed_pass(profile):
        sess.mla.set_option(B.MLA_OPT_PROFILE, 1 if profile else 0)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        kms = []
        for a, z in ev:
            flush_l2()
            a.record(stream)
            step()
            z.record(stream)
            if profile:
                kms.append(sess.mla.profile_read())
        torch.cuda.synchronize()
        return [a.elapsed_time(z) for a, z in ev], kms

    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    step_ms, _ = timed_pass(False)
    torch.cuda.synchronize()
    _, kernel_ms = timed_pass(True)
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    sess.mla.set_option(B.MLA_OPT_PROFILE, 0)
    if sess.status() != 0:
        raise SystemExit("device check word set during the timed steps")
    ms = statistics.mean(step_ms)

    # end to end with host buffers: the prompt rows, indices and queries in, the outputs back
    parts = [("rows", wl.rows.view(np.int16)), ("seq", wl.row_seq.astype(np.int32)),
             ("pos", wl.row_pos.astype(np.int32)), ("q", p["q"].view(np.int16)),
             ("q_start", p["q_start"].astype(np.int32)), ("q_len", p["q_len"].astype(np.int32)),
             ("ctx", wl.ctx_len.astype(np.int32))]
    offs, total = {}, 0
    for name, a in parts:
        offs[name] = total
        total += (a.nbytes + 255) // 256 * 256
    h_pack = torch.empty(total, dtype=torch.uint8).pin_memory()
    d_pack = torch.empty(total, dtype=torch.uint8, device=dev)
    views = {}
    for name, a in parts:
        flat = np.ascontiguousarray(a).reshape(-1)
        h_pack[offs[name]:offs[name] + flat.nbytes].copy_(torch.from_numpy(flat.view(np.uint8)))
        dt = torch.int16 if flat.dtype == np.int16 else torch.int32
        views[name] = d_pack[offs[name]:offs[name] + flat.nbytes].view(dt).view(a.shape)
    h_out = torch.empty(tuple(out.shape), dtype=torch.int16).pin_memory()
    h2d = sum(a.nbytes for _, a in parts)
    d2h = h_out.numel() * 2

    def e2e_step():
        d_pack.copy_(h_pack, non_blocking=True)
        step(views["rows"].view(torch.bfloat16), views["seq"], views["pos"], views["q"].view(torch.bfloat16),
             views["q_start"], views["q_len"], views["ctx"])
        h_out.copy_(out.view(torch.int16), non_blocking=True)

    for _ in range(max(1, args.warmup)):
        flush_l2()
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(args.steps):
        flush_l2()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        z.record(stream)
        z.synchronize()
        e2e_ms.append(a.elapsed_time(z))
    e2e_serial = statistics.mean(e2e_ms)
    d_packs = [d_pack, torch.empty_like(d_pack)]
    views_k = [views, {}]
    for name, a in parts:
        n = np.ascontiguousarray(a).nbytes
        dt = torch.int16 if np.asarray(a).dtype == np.int16 else torch.int32
        views_k[1][name] = d_packs[1][offs[name]:offs[name] + n].view(dt).view(a.shape)
    outs = [out, torch.empty_like(out)]
    h_outs = [h_out, torch.empty_like(h_out).pin_memory()]

    def slot_step(k):
        v = views_k[k]
        step(v["rows"].view(torch.bfloat16), v["seq"], v["pos"], v["q"].view(torch.bfloat16), v["q_start"],
             v["q_len"], v["ctx"], outs[k])
    e2e = pipelined_e2e(stream, dev, h_pack, d_packs, outs, h_outs, slot_step, args.steps, args.warmup)

    ms, e2e = ranks_max([ms, e2e], dev, world)
    fe, fa = prefill_flops(wl)
    hbm, tc_burst, tc_sust, peak_kind = peaks()
    per_kernel = {k: round(statistics.mean(km[k] for km in kernel_ms) * 1000.0, 2) for k in kernel_ms[0]}
    attn_ms = per_kernel["mla_prefill_attention"] / 1000.0
    exp_ms = per_kernel["mla_prefill_expand"] / 1000.0
    achieved = fa / (attn_ms * 1e-3) / 1e12
    if rank == 0:
        line = {
            "metric": PREFILL_METRIC, "value": round(job_rate(world, fe + fa, ms) / 1e12, 2), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "us_per_step": round(ms * 1000.0, 2), "us_per_step_median": round(statistics.median(step_ms) * 1000.0, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.B, "s_ctx": wl.max_ctx, "n_h": wl.n_h, "q_len": max_q,
                       "mode": "MHA (latent expanded per head), causal, whole prompts",
                       "flops_per_step": {"expansion": int(fe), "attention": int(fa)},
                       "l2": f"flushed between steps outside the timed events ({flush.numel() >> 20} MiB write + "
                             f"read); the step's queries ({q.numel() * 2 >> 20} MiB) also exceed L2",
                       "timing": "value from K steps without per-kernel events; per_kernel_us and roofline from "
                                 "a second K-step pass with per-kernel events",
                       "arithmetic": "bf16 MMA operands (expanded K/V, P), fp32 accumulation and softmax",
                       "parallelism": f"replicas x{world}"},
            "per_kernel_us": per_kernel,
            "roofline": {"bound": "tensor", "kernel": "mla_prefill_attention", "achieved": round(achieved, 1),
                         "peak": tc_burst, "unit": "TFLOP/s", "frac": round(achieved / tc_burst, 4),
                         "traffic": ncu_traffic(wl, "prefill_traffic.json", PREFILL_SOURCES),
                         "peak_source": f"{peak_kind} bf16_tflops (burst)",
                         "algorithmic_flops_per_launch": int(fa),
                         "expansion": {"achieved": round(fe / (exp_ms * 1e-3) / 1e12, 1),
                                       "frac": round(fe / (exp_ms * 1e-3) / 1e12 / tc_burst, 4)}},
            "e2e": {"value": round(job_rate(world, fe + fa, e2e) / 1e12, 2), "unit": "TFLOP/s",
                    "ms_per_step": round(e2e, 5), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "mode": E2E_MODE, "serial_ms_per_step": round(e2e_serial, 5)},
            "gpu_launches": args.steps * 3,
            "clocks": clock_info,
        }
        if world == 1 and not args.no_cpu_baseline:
            v, _, desc = prefill_oracle_sample(wl, args.cpu_seconds)
            line["cpu_baseline"] = {"value": round(v, 6), "unit": "TFLOP/s", "cores": blas_threads(),
                                    "kind": "oracle", "sample": desc}
        print(json.dumps(line), flush=True)
    sess.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference" and int(os.environ.get("RANK", "0")) != 0:
        return 0                             # the reference arm runs on rank 0 alone
    if args.workload == PREFILL:
        wl = workload(args.workload)
        if args.impl == "reference":
            return run_prefill_reference(args, wl)
        return run_prefill(args, wl)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
