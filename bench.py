"""Benchmark of the speculative-decoding verify step on GB300.

One step = the whole hot path on one batch: kv_append -> spec_verify_attn ->
spec_rejection_sample -> kv_rollback, four C-ABI calls on one stream.

Default workload: the Llama-3-8B-shaped batch (32 sequences, contexts
U[512, 4096], K = 5, 32 q / 8 kv heads of dim 128, bf16 KV in 16-token
blocks, vocab 128256, T = 1). The cache state evolves from step to step like
a decode loop (each step keeps a_b + 1 tokens per sequence). Two input sets
(logits, drafts, uniforms, new rows and queries) alternate from step to step,
so a step's 92 MB of sampler inputs were last read two steps before, with more
than 700 MB of other traffic in between (L2: 129 MB). A set's decisions depend
on its inputs alone, so the tokens each step keeps, and the bytes each step
reads, are known exactly.

The line also carries `configs`: the same measurements on the other workloads
(Llama-8B shape greedy, Llama-70B shape at T = 1 and greedy, the
continuous-batching mix, the draft trees greedy and at T = 1).

Prints one JSON line. `--impl reference` times the fp64 CPU oracle on the
host cores instead (bounded samples of the same workload). `--profile
attention|sampler` runs only that call of the default workload six times (for
a profiler's capture) and prints nothing else.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "spec-verify seqs/s & tokens/s; achieved HBM TB/s vs 8 TB/s (1 GB300)"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
PROFILES = os.path.join(ROOT, "profiles")
ATTN_SOURCES = ["attn_umma.cu", "sv_internal.cuh"]  # the files that define attn_umma_kernel
SAMPLER_SOURCES = ["sampler.cu", "sv_internal.cuh"]  # the files that define the sampler's kernels


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--config", default="llama8b", choices=["llama8b", "llama70b", "contbatch", "tree"])
    p.add_argument("--temperature", type=float, default=1.0)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--no-configs", action="store_true")
    p.add_argument("--profile", choices=["attention", "sampler"], default=None)
    return p.parse_args()


# ----------------------------------------------------------------------------
# workload
# ----------------------------------------------------------------------------
def make_case(name, temperature, steps_total, seed_offset=0):
    from speculative_decoding_verify_paged_gb300 import workloads as W
    if name == "llama8b":
        case = W.llama8b(seed=1 + seed_offset, temperature=temperature, growth_tokens=6 * steps_total)
        desc = ("llama3-8b-shaped verify: B=32, ctx U[512,4096], K=5, 32q/8kv heads, head_dim 128, bf16 KV "
                "in 16-token blocks (shuffled pool), vocab 128256, bf16 logits, T=%g" % temperature)
    elif name == "llama70b":
        case = W.llama70b(seed=2 + seed_offset, temperature=temperature)
        desc = "llama3-70b-shaped verify: B=128, ctx U[512,640], K=4, 64q/8kv, bf16, bs16, vocab 128256"
    elif name == "contbatch":
        case = W.contbatch(seed=3 + seed_offset)
        desc = "continuous-batching mix: B=256, lognormal ctx, K_b U{2..8}, bs128, fragmented pool"
    else:
        case = W.tree(seed=5 + seed_offset)
        desc = "tree verify: B=16, ctx 8192, 61 rows (60-node tree), bs64, vocab 32000, greedy"
    return case, desc


def second_inputs(name, case, temperature, seed_offset=0):
    """Another input set of the workload's shapes (the main loop alternates the two);
    None where the workload has one (the sets of the continuous-batching mix and of
    the trees differ in shape)."""
    from speculative_decoding_verify_paged_gb300 import workloads as W
    if name == "llama8b":
        return W.llama8b_step(1 + seed_offset, 1, temperature=temperature)
    if name == "llama70b":
        return W.llama70b_step(2 + seed_offset, 1, temperature=temperature)
    return None


def attn_bytes(ctx_plus_n, step, state):
    """Algorithmic bytes of one attention launch: every visible K and V row once,
    Q in, O out."""
    el = {"bf16": 2, "e4m3": 1}.get(state.dtype, 4)  # pool element
    io = 4 if state.dtype == "f32" else 2  # an fp8 pool takes bf16 queries and outputs
    kv = int(ctx_plus_n.sum()) * 2 * state.num_kv_heads * state.head_dim * el
    qo = 2 * step.total_q * step.num_q_heads * state.head_dim * io
    return kv + qo


def sampler_bytes(step):
    el = 2 if step.logits_dtype == "bf16" else 4
    rows = step.total_q if step.temperature == 0.0 or step.mask_kind == "tree" else 2 * step.total_q - len(step.n_q)
    return rows * step.vocab * el


def attn_flops(ctx, step, G):
    # 4 * Hq * D * sum_b n_b * (c_b + (n_b + 1) / 2) for causal rows
    n = step.n_q.astype(np.float64)
    return float(4 * step.num_q_heads * step.q.shape[-1] * (n * (ctx + (n + 1) / 2)).sum())


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, enabled: bool):
        self.proc = None
        self.path = None
        if not enabled:
            return
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------
# CPU oracle timing
# ----------------------------------------------------------------------------
def oracle_sample_step(case, seqs):
    """The oracle's verify step restricted to the sequences `seqs`: append, fp64
    attention, sampler (or tree walk), rollback. Returns the seconds it took.
    The oracle writes the appended rows straight into the case's host pools
    (the same rows into the same free blocks on every call)."""
    import oracle
    from speculative_decoding_verify_paged_gb300 import workloads as W
    st, sp = case.state, case.step
    seqs = np.asarray(seqs, np.int64)
    sub = W.KVState(st.block_size, st.num_blocks, st.max_blocks_per_seq, st.num_kv_heads, st.head_dim, st.dtype,
                    st.k_pool, st.v_pool, st.block_table[seqs].copy(), st.seq_lens[seqs].copy(),
                    st.free_list.copy(), st.free_top)
    n_q = sp.n_q[seqs]
    cu = np.concatenate([[0], np.cumsum(n_q)]).astype(np.int32)
    rows = np.concatenate([np.arange(sp.cu_q[b], sp.cu_q[b + 1]) for b in seqs])
    drows = np.concatenate([np.arange(sp.cu_q[b] - b, sp.cu_q[b + 1] - b - 1) for b in seqs]).astype(np.int64)
    sub_step = W.StepInputs(n_q, cu, sp.num_q_heads, sp.q[rows], sp.new_k[rows], sp.new_v[rows], sp.vocab,
                            sp.logits_dtype, sp.target_logits[rows], sp.draft_logits[drows],
                            sp.draft_tokens[drows], sp.u_accept[drows], sp.u_resample[seqs], sp.temperature,
                            sp.mask_kind, None if sp.tree_mask is None else sp.tree_mask[rows],
                            None if sp.parent is None else sp.parent[rows])
    okv = oracle.OracleKV(sub, with_pools=False)
    okv.k_pool, okv.v_pool = st.k_pool, st.v_pool
    t0 = time.perf_counter()
    assert okv.append(sub_step) is None
    oracle.paged_attention(okv.as_state(), sub_step)
    if sp.mask_kind == "tree":
        r = oracle.tree_greedy(sub_step)
        okv.rollback(sub_step, r.accept_cnt, path_nodes=r.path_nodes)
    else:
        r = oracle.rejection_sample(sub_step)
        okv.rollback(sub_step, r.accept_cnt)
    return time.perf_counter() - t0


def cpu_seqs_for(case, budget_s=15.0):
    """How many sequences of the batch fit the CPU budget (estimated from one)."""
    t1 = oracle_sample_step(case, [0])
    n = max(1, min(case.state.batch, int(budget_s / max(t1, 1e-3))))
    return n, t1


# ----------------------------------------------------------------------------
# native arm
# ----------------------------------------------------------------------------
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def traffic_record(name, sources):
    """A kernel's DRAM traffic from a committed ncu summary, valid only while the
    kernel's sources are unchanged (matching hash)."""
    path = os.path.join(PROFILES, name)
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    h = hashlib.sha256()
    for src in sources:
        h.update(open(os.path.join(ROOT, "speculative_decoding_verify_paged_gb300", "csrc", src), "rb").read())
    return rec if rec.get("sources_sha256") == h.hexdigest() else None


def aggregate(elapsed_ms: float, seqs_local: int, world: int, device=None):
    """Whole-job throughput over the ranks of the default process group: the
    slowest rank's time, the sum of the sequences every rank verified."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    n = torch.tensor([seqs_local], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(n, op=dist.ReduceOp.SUM)
    ms = float(t.item())
    return float(n.item()) / (ms / 1e3), ms


class StepLoop:
    """The verify step of one workload on the device, with its input sets: the
    cache state, one DeviceStep per input set (used in turn), shared buffers,
    and the tokens each set keeps per sequence (a_b + 1, from a first run: a
    set's decisions depend on its inputs alone), so that the context lengths,
    and the bytes every step reads, are known without reading the device."""

    def __init__(self, state, sets, growth, dev):
        from speculative_decoding_verify_paged_gb300 import step as S
        self.S = S
        self.state, self.sets = state, sets
        self.kv = S.device_kv(state, dev)
        self.ds = [S.DeviceStep.from_host(x, dev) for x in sets]
        self.msl = int(max((state.seq_lens + x.n_q).max() for x in sets)) + growth + 16
        big = max(range(len(sets)), key=lambda k: (sets[k].max_q, sets[k].total_q))
        self.buf = S.StepBuffers.make(self.kv, self.ds[big], self.msl, dev)
        self.keep = [None] * len(sets)
        self.lens = state.seq_lens.astype(np.int64).copy()  # the host's copy of the committed lengths
        self.count = 0  # steps run

    def step(self, stream, ev=None):
        """One step with the next input set; `ev` (three events) brackets attention and sampler."""
        S, k = self.S, self.count % len(self.ds)
        d, buf = self.ds[k], self.buf
        S.append(self.kv, d, buf, stream)
        if ev is not None:
            ev[0].record(stream)
        S.attention(self.kv, d, buf, self.msl, stream)
        if ev is not None:
            ev[1].record(stream)
        S.sample(d, buf, stream)
        if ev is not None:
            ev[2].record(stream)
        S.rollback(self.kv, d, buf, stream)
        self.count += 1
        return k

    def learn(self, stream):
        """One step with every set, reading back the tokens each keeps."""
        import torch
        for _ in range(len(self.ds)):
            before = self.kv.seq_lens.clone()
            k = self.step(stream)
            torch.cuda.synchronize()
            assert int(self.buf.status.item()) == 0, "device status set"
            self.keep[k] = (self.kv.seq_lens - before).cpu().numpy().astype(np.int64)
            self.lens += self.keep[k]

    def advance(self, k):
        """The host's lengths after a step of set k; returns the lengths that step started from."""
        c = self.lens.copy()
        self.lens += self.keep[k]
        return c

    def attn_bytes_flops(self, c, k):
        x = self.sets[k]
        G = x.num_q_heads // self.state.num_kv_heads
        return attn_bytes(c + x.n_q, x, self.state), attn_flops(c, x, G)


def timed_loop(loop, steps, stream, per_call):
    """`steps` steps back to back (per_call: with events around attention and the
    sampler); returns the total ms, the per-call ms lists, and per step the
    attention bytes and flops, the sampler bytes and the emitted tokens."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)] if per_call else None
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ab, fl, sb, em = [], [], [], []
    torch.cuda.synchronize()
    t0.record(stream)
    for s in range(steps):
        k = loop.step(stream, evs[s] if per_call else None)
        c = loop.advance(k)
        b, f = loop.attn_bytes_flops(c, k)
        ab.append(b)
        fl.append(f)
        sb.append(sampler_bytes(loop.sets[k]))
        em.append(int(loop.keep[k].sum()))
    t1.record(stream)
    torch.cuda.synchronize()
    assert int(loop.buf.status.item()) == 0, "device status set during the timed steps"
    attn_ms = [e[0].elapsed_time(e[1]) for e in evs] if per_call else None
    samp_ms = [e[1].elapsed_time(e[2]) for e in evs] if per_call else None
    return t0.elapsed_time(t1), attn_ms, samp_ms, ab, fl, sb, em


def run_native(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    # every step this run takes (the learning steps, warm-up, the timed pass, the per-call pass,
    # the path timings, the end-to-end leg): each keeps at most K + 1 = 6 tokens a sequence,
    # and the cache is sized for it
    steps_total = 2 + args.warmup + 2 * args.steps + 2 + max(3, args.warmup) + max(10, args.steps // 2) + 2
    case, desc = make_case(args.config, args.temperature, steps_total, seed_offset=rank)
    st, sp = case.state, case.step
    second = second_inputs(args.config, case, args.temperature, seed_offset=rank)
    sets = [sp] if second is None else [sp, second]
    growth = 6 * steps_total if args.config == "llama8b" else 0
    loop = StepLoop(st, sets, growth, dev)
    kv, d, buf, msl = loop.kv, loop.ds[0], loop.buf, loop.msl
    stream = torch.cuda.current_stream(dev)
    loop.learn(stream)
    for _ in range(args.warmup):
        loop.advance(loop.step(stream) % len(sets))
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0, "device status set during warm-up"

    if args.profile:
        # only the one call, six times, on the state the warm-up left (the append of the
        # attention's rows done once); nothing printed
        S = loop.S
        S.append(kv, d, buf, stream)
        for _ in range(6):
            if args.profile == "attention":
                S.attention(kv, d, buf, msl, stream)
            else:
                S.sample(d, buf, stream)
        torch.cuda.synchronize()
        assert int(buf.status.item()) == 0
        return

    # the timed pass: K steps back to back, nothing recorded between the calls (an event
    # between two kernels ends the programmatic dependent launch that lets each kernel's
    # start overlap the previous one's end)
    clocks = Clocks(local, not args.no_clocks and rank == 0)
    if world > 1:
        dist.barrier()
    elapsed_ms, _, _, _, _, sb_t, em_t = timed_loop(loop, args.steps, stream, per_call=False)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    emitted = int(np.sum(em_t))

    # the per-call pass: K more steps with events around the attention and sampler calls
    _, attn_ms, samp_ms, ab, fl, sb, _ = timed_loop(loop, args.steps, stream, per_call=True)
    # near-ties of the last step's decisions: sequences whose smallest |uniform - threshold| is below
    # 1e-4 (+inf at T = 0 or for greedy trees)
    near_ties = int((buf.margin < 1e-4).sum().item()) if sp.temperature > 0 else 0
    attn_bytes_avg = float(np.mean(ab))
    attn_ms_avg = float(np.mean(attn_ms))
    samp_ms_avg = float(np.mean(samp_ms))
    samp_bytes_avg = float(np.mean(sb))

    B = st.batch
    value, elapsed_ms = aggregate(elapsed_ms, B * args.steps, world, dev)

    paths = attn_path_times(kv, d, buf, msl, stream)
    e2e = None if args.no_e2e else run_e2e(args, kv, d, buf, msl, sp, dev, stream, world)
    hbm_peak, peak_kind = peaks()
    achieved = attn_bytes_avg / (attn_ms_avg / 1e3) / 1e9
    traffic = traffic_record("attn_traffic.json", ATTN_SOURCES)
    samp_traffic = traffic_record("sampler_traffic.json", SAMPLER_SOURCES)
    line = {
        "metric": METRIC, "value": value, "unit": "seqs/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if st.dtype == "bf16" else "f32",
        "data": "synthetic (seeded numpy PCG64; no dataset or weights)",
        "config": {"workload": desc, "global_batch": B * world, "scored_tokens_per_step": sp.total_q,
                   "l2": ("inputs larger than L2 (129 MB): each step streams the whole KV prefix (>300 MB) and "
                          "the logits; %d input sets alternate, so a step's logits were last read %d steps "
                          "before" % (len(sets), len(sets))),
                   "input_sets": len(sets), "state": "cache evolves across steps (a_b+1 tokens kept)",
                   "timing": "value: K steps with nothing recorded between the calls; roofline and "
                             "sampler_roofline per-call times: K further steps with CUDA events around "
                             "each call (the events cut the programmatic overlap between kernels)"},
        "tokens_per_s": emitted * world / (elapsed_ms / 1e3),
        "scored_tokens_per_s": sp.total_q * args.steps * world / (elapsed_ms / 1e3),
        "mean_tokens_per_seq_step": emitted / (B * args.steps),
        "roofline": {"kernel": "spec_verify_attn (persistent tcgen05 attention + combine)", "bound": "hbm",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS, "peak_source": peak_kind,
                     "traffic": (traffic["traffic_per_algorithmic_byte"] * attn_bytes_avg if traffic else None),
                     "tensor_pipe_active": traffic.get("tensor_pipe_active_pct") if traffic else None,
                     "algorithmic_bytes_per_launch": attn_bytes_avg, "avg_launch_ms": attn_ms_avg,
                     "tflops": float(np.mean(fl)) / (attn_ms_avg / 1e3) / 1e12},
        "sampler_roofline": {"kernel": "spec_rejection_sample (statistics + decisions)", "bound": "hbm",
                             "achieved": samp_bytes_avg / (samp_ms_avg / 1e3) / 1e9, "peak": hbm_peak,
                             "unit": "GB/s", "frac": samp_bytes_avg / (samp_ms_avg / 1e3) / 1e9 / hbm_peak,
                             "traffic": (samp_traffic["traffic_per_algorithmic_byte"] * samp_bytes_avg
                                         if samp_traffic else None),
                             "algorithmic_bytes_per_launch": samp_bytes_avg, "avg_launch_ms": samp_ms_avg},
        "hbm_gbs_step": (float(np.mean(ab)) + float(np.mean(sb_t))) / (elapsed_ms / args.steps / 1e3) / 1e9,
        "near_ties": {"sequences_per_step": near_ties, "of": B, "threshold": 1e-4,
                      "note": "sampler margin output: decisions within 1e-4 of their threshold"},
        "attn_paths_ms": paths,
        "gpu_launches": S_launches(loop) * args.steps,
        "clocks": clk,
        "adaptive_k": adaptive_k_timing(),
        "cow": cow_timing(),
        "tree_sampler": tree_sampler_timing(hbm_peak),
        "fp8_kv": fp8_timing(hbm_peak),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_configs and rank == 0:
        del loop, kv, d, buf
        torch.cuda.empty_cache()
        line["configs"] = config_records(hbm_peak, dev, stream)
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(case, B)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


def S_launches(loop):
    return loop.S.launches_per_step(loop.ds[0], loop.msl, loop.kv)


def cpu_baseline(case, B):
    """The fp64 oracle's verify step on the host cores: a bounded sample of the bench's
    workload on one thread and on every core, and, per workload, one timed step
    (the continuous-batching mix: one of its ten iterations, times ten)."""
    import oracle
    from speculative_decoding_verify_paged_gb300 import workloads as W
    cores = os.cpu_count() or 1
    oracle.set_threads(1)
    n, t1 = cpu_seqs_for(case, budget_s=10.0)
    seqs = list(range(n))
    t_one = oracle_sample_step(case, seqs)
    used = oracle.set_threads(cores)  # OpenMP over (sequence, KV head) and sequences; same values
    t_all = oracle_sample_step(case, seqs)
    out = {"value": n / t_all, "unit": "seqs/s", "cores": used, "kind": "oracle",
           "sample": f"one verify step of {n} of the {B} sequences (fp64 C oracle: append, "
                     f"attention, sampler, rollback), {t_all:.1f} s on {used} threads",
           "single_thread": {"value": n / t_one, "cores": 1, "seconds": t_one}}
    per = {}
    for name in ("tiny", "llama8b", "llama70b", "contbatch", "tree"):
        c = W.CONFIGS[name]()
        bsz = c.state.batch
        secs = oracle_sample_step(c, list(range(bsz)))
        rec = {"seqs_per_s": bsz / secs, "seconds": secs, "sequences": bsz, "threads": used}
        if name == "contbatch":
            rec["note"] = ("one iteration timed; the 10-iteration loop extrapolated: %.1f s" % (10 * secs))
            rec["extrapolated_10_iterations_s"] = 10 * secs
        per[name] = rec
        del c
    out["configs"] = per
    return out


CONFIG_RUNS = (("llama8b", 0.0), ("llama70b", 1.0), ("llama70b", 0.0), ("contbatch", 1.0), ("tree", 0.0),
               ("tree", 1.0))


def config_records(hbm_peak, dev, stream, steps=10, warmup=2):
    """Per workload: `steps` steps back to back (seqs/s, tokens/s), then `steps` with
    events around attention and the sampler (their HBM fractions); input sets in turn
    (two for the fixed-shape workloads; three iterations of the continuous-batching
    mix, whose K_b are redrawn each iteration; the trees have one)."""
    import torch
    from speculative_decoding_verify_paged_gb300 import workloads as W
    out = {}
    for name, T in CONFIG_RUNS:
        total = 3 + warmup + 2 * steps
        if name == "llama8b":
            case = W.llama8b(temperature=T, growth_tokens=6 * total)
            sets = [case.step, W.llama8b_step(1, 1, temperature=T)]
        elif name == "llama70b":
            case = W.llama70b(temperature=T, growth_tokens=5 * total)
            sets = [case.step, W.llama70b_step(2, 1, temperature=T)]
        elif name == "contbatch":
            case = W.contbatch(iterations=total)
            sig = case.meta["sigma_b"]
            sets = [case.step] + [W.contbatch_step(3, it, batch=case.state.batch, vocab=case.step.vocab, sigma_b=sig)
                                  for it in (1, 2)]
        else:
            case = W.tree(temperature=T, growth_tokens=7 * total)
            sets = [case.step]
        growth = {"llama8b": 6, "llama70b": 5, "contbatch": 9, "tree": 7}[name] * total
        loop = StepLoop(case.state, sets, growth, dev)
        loop.learn(stream)
        for _ in range(warmup):
            loop.advance(loop.step(stream) % len(sets))
        ms, _, _, _, _, _, em = timed_loop(loop, steps, stream, per_call=False)
        _, attn_ms, samp_ms, ab, fl, sb, _ = timed_loop(loop, steps, stream, per_call=True)
        B = case.state.batch
        a_ms, s_ms = float(np.mean(attn_ms)), float(np.mean(samp_ms))
        a_gbs = float(np.mean(ab)) / (a_ms / 1e3) / 1e9
        s_gbs = float(np.mean(sb)) / (s_ms / 1e3) / 1e9
        rec = {"seqs_per_s": B * steps / (ms / 1e3), "tokens_per_s": float(np.sum(em)) / (ms / 1e3),
               "scored_tokens_per_s": float(np.mean([x.total_q for x in sets])) * steps / (ms / 1e3),
               "ms_per_step": ms / steps, "input_sets": len(sets), "steps": steps,
               "attention": {"ms": a_ms, "bytes": float(np.mean(ab)), "achieved_gbs": a_gbs, "frac": a_gbs / hbm_peak,
                             "tflops": float(np.mean(fl)) / (a_ms / 1e3) / 1e12},
               "sampler": {"ms": s_ms, "bytes": float(np.mean(sb)), "achieved_gbs": s_gbs, "frac": s_gbs / hbm_peak},
               "near_ties": (int((loop.buf.margin[:B] < 1e-4).sum().item()) if T > 0 else 0)}
        out[f"{name}_T{T:g}"] = rec
        del loop, case, sets
        torch.cuda.empty_cache()
    return out


def tree_sampler_timing(hbm_peak, reps=20):
    """The tree sampler on the draft-tree workload (16 trees of 60 nodes + root,
    V = 32000 bf16): greedy (sv_tree_greedy_accept) and lossless at T = 1
    (sv_tree_rejection_sample). Device time per call, CUDA events; before each
    call the L2 is emptied of the logits by reading a 256 MB buffer ("read"),
    and, as a second figure, by writing it ("write": the call then also pays for
    evicting 129 MB of dirty lines); the median of the reps; bytes = every
    target row once."""
    import torch
    from speculative_decoding_verify_paged_gb300 import step as S
    from speculative_decoding_verify_paged_gb300 import workloads as W
    out = {}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for name, T in (("greedy", 0.0), ("t1", 1.0)):
        case = W.tree(temperature=T)
        d = S.DeviceStep.from_host(case.step)
        kv = S.device_kv(case.state)
        buf = S.StepBuffers.make(kv, d, int((case.state.seq_lens + case.step.n_q).max()))
        S.sample(d, buf)
        times = {}
        for how in ("read", "write"):
            ms = []
            for _ in range(reps):
                if how == "read":
                    flush.max()
                else:
                    flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                S.sample(d, buf)
                b.record()
                torch.cuda.synchronize()
                ms.append(a.elapsed_time(b))
            times[how] = float(np.median(ms))  # median: a rep can catch the flush's own tail
        t = times["read"]
        nbytes = case.step.target_logits.shape[0] * case.step.vocab * 2
        out[name] = {"us": t * 1e3, "us_after_dirty_flush": times["write"] * 1e3, "bytes": int(nbytes),
                     "achieved_gbs": nbytes / (t / 1e3) / 1e9, "frac": nbytes / (t / 1e3) / 1e9 / hbm_peak,
                     "status": int(buf.status.item())}
        del kv, buf, d
    return out


def fp8_timing(hbm_peak, steps=5, warmup=3):
    """Verify steps of the Llama-8B-shaped batch (32 sequences, K = 5, T = 1) on
    an E4M3 KV pool: append (quantising), attention (the tcgen05 kernel with its
    code-widening warps; the CUDA-core kernel timed beside it), sampler,
    rollback. CUDA events per kernel group, averaged over the timed steps;
    attention bytes = every visible K and V code once, bf16 Q in and O out."""
    import torch
    from speculative_decoding_verify_paged_gb300 import step as S
    from speculative_decoding_verify_paged_gb300 import workloads as W
    case = W.llama8b(growth_tokens=6 * (steps + warmup + 2), kv_dtype="e4m3")
    st, sp = case.state, case.step
    msl = int((st.seq_lens + sp.n_q).max()) + 6 * (steps + warmup + 2) + 16
    kv = S.device_kv(st)
    d = S.DeviceStep.from_host(sp)
    buf = S.StepBuffers.make(kv, d, msl)
    for _ in range(warmup):
        S.append(kv, d, buf)
        S.attention(kv, d, buf, msl)
        S.sample(d, buf)
        S.rollback(kv, d, buf)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    lens = []
    for s in range(steps):
        lens.append(kv.seq_lens.cpu().numpy().astype(np.int64))
        ev[s][0].record()
        S.append(kv, d, buf)
        ev[s][1].record()
        S.attention(kv, d, buf, msl)
        ev[s][2].record()
        S.sample(d, buf)
        S.rollback(kv, d, buf)
        ev[s][3].record()
        torch.cuda.synchronize()
    attn = float(np.mean([e[1].elapsed_time(e[2]) for e in ev]))
    step_ms = float(np.mean([e[0].elapsed_time(e[3]) for e in ev]))
    paths = attn_path_times(kv, d, buf, msl, torch.cuda.current_stream(), reps=5,
                            names=("tensor_cores", "cuda_cores"))
    nbytes = float(np.mean([attn_bytes(c + sp.n_q, sp, st) for c in lens]))
    out = {"workload": "llama8b shape, E4M3 KV pool (scale 0.125), T = 1", "step_us": step_ms * 1e3,
           "attention_us": attn * 1e3, "attention_bytes": nbytes,
           "attention_achieved_gbs": nbytes / (attn / 1e3) / 1e9,
           "attention_frac": nbytes / (attn / 1e3) / 1e9 / hbm_peak, "attn_paths_ms": paths,
           "status": int(buf.status.item())}
    del kv, buf, d
    return out


def cow_timing(reps=5):
    """Copy-on-write sharing through the C ABI (parallel sampling): 8 sequences
    with llama8b-shaped contexts (16-token blocks, 8 KV heads of 128 bf16) fork
    into 3 children each; then one append of a verify step (K=5) for all 32,
    where every shared partial last block is copied by all but its last writer;
    then the children are released. Device time of each call, CUDA events, mean
    over `reps` rounds."""
    import torch
    from speculative_decoding_verify_paged_gb300 import _lib as L
    from speculative_decoding_verify_paged_gb300 import step as S
    from speculative_decoding_verify_paged_gb300 import workloads as W
    P, C = 8, 3
    B = P * (C + 1)
    rng = np.random.default_rng(7)
    ctx = np.zeros(B, np.int32)
    ctx[:P] = rng.integers(512, 4097, size=P)
    st = W.make_kv_state(7, ctx, block_size=16, num_kv_heads=8, head_dim=128, dtype="bf16",
                         growth_tokens=8 * reps + 16)
    ref = np.zeros(st.num_blocks, np.int32)
    for b in range(B):
        ref[st.block_table[b, :(int(ctx[b]) + 15) // 16]] = 1
    kv = S.device_kv(st, ref_count=ref)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    parents = torch.arange(P, dtype=torch.int32, device="cuda").repeat_interleave(C)
    children = torch.arange(P, B, dtype=torch.int32, device="cuda")
    step = W.make_chain_step(7, np.full(B, 6, np.int32), num_q_heads=32, num_kv_heads=8, head_dim=128,
                             qkv_dtype="bf16", vocab=256, logits_dtype="bf16", target_sigma=3.0, draft_coef=0.8,
                             draft_sigma=1.0, temperature=0.0)
    d = S.DeviceStep.from_host(step)
    accept = torch.zeros(B, dtype=torch.int32, device="cuda")
    times = {"fork": [], "append_with_copies": [], "release": []}
    copies = 0
    lens = ctx[:P].astype(np.int64)
    for r in range(reps):
        copies += int(sum(C for b in range(P) if lens[b] % 16))  # the last of the C + 1 writers writes in place
        lens += 1  # rollback keeps one row of each sequence (a = 0)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        torch.cuda._sleep(2_000_000)  # keeps the GPU busy while the host queues the calls: no launch gaps timed
        ev[0].record()
        L.kv_fork(kv, parents, children, status)
        ev[1].record()
        ev[2].record()
        L.kv_append(kv, d.new_k, d.new_v, d.cu_q, status)
        ev[3].record()
        L.kv_rollback(kv, d.cu_q, accept, status, max_q=6)
        ev[4].record()
        L.kv_release(kv, children, status)
        ev[5].record()
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            return {"error": L.status_string(int(status.item()))}
        times["fork"].append(ev[0].elapsed_time(ev[1]) * 1e3)
        times["append_with_copies"].append(ev[2].elapsed_time(ev[3]) * 1e3)
        times["release"].append(ev[4].elapsed_time(ev[5]) * 1e3)
    out = {k + "_us": float(np.mean(v)) for k, v in times.items()}
    out.update({"sequences": B, "forked_pairs": P * C, "block_copies_per_append": copies / reps,
                "note": "sv_kv_fork / sv_kv_append / sv_kv_release with ref_count, device time"})
    return out


def adaptive_k_timing(batch=256, calls=2000):
    """Host cost of the adaptive-K controller (sv_adaptive_k_update through the
    C ABI) for a 256-sequence batch with a full 50-rate window."""
    from speculative_decoding_verify_paged_gb300 import AdaptiveK
    rng = np.random.default_rng(0)
    ctl = AdaptiveK(batch)
    drafted = np.full(batch, 8, np.int32)
    acc = [rng.integers(0, 9, size=batch).astype(np.int32) for _ in range(16)]
    for i in range(60):
        ctl.update(acc[i % 16], drafted)
    t0 = time.perf_counter()
    for i in range(calls):
        ctl.update(acc[i % 16], drafted)
    us = (time.perf_counter() - t0) / calls * 1e6
    return {"call": "sv_adaptive_k_update", "batch": batch, "window": 50, "us_per_update": us,
            "note": "host-side, once per step between sampler and the next append"}


def attn_path_times(kv, d, buf, msl, stream, reps=10, names=("keys_major", "tensor_cores", "warp_mma", "cuda_cores")):
    """The attention call alone, timed with each implementation on the same cache
    state (the step's rows appended once, rolled back after)."""
    import torch
    from speculative_decoding_verify_paged_gb300 import _lib as L
    from speculative_decoding_verify_paged_gb300 import step as S
    out = {}
    S.append(kv, d, buf, stream)
    for path in names:
        try:
            L.set_attn_path(path)
            for _ in range(2):
                S.attention(kv, d, buf, msl, stream)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                S.attention(kv, d, buf, msl, stream)
            b.record(stream)
            torch.cuda.synchronize()
            out[path] = a.elapsed_time(b) / reps
        except L.SVError:
            out[path] = None
        finally:
            L.set_attn_path("auto")
    S.sample(d, buf, stream)
    S.rollback(kv, d, buf, stream)
    torch.cuda.synchronize()
    return out


def run_e2e(args, kv, d, buf, msl, sp, dev, stream, world):
    """The same step through the public API with the step's inputs in pinned host
    memory: H2D of the inputs, the four calls, D2H of the results, every step.
    Two input buffers: the inputs of step i + 1 are copied on a second stream
    while step i computes, as a serving loop would overlap them."""
    import torch
    from speculative_decoding_verify_paged_gb300 import step as S
    host = S.DeviceStep.tensors_of(sp, lambda x: S._host(x, pin=True))
    names = [k for k, v in host.items() if v is not None]
    h2d = sum(host[k].numel() * host[k].element_size() for k in names)
    d2 = S.DeviceStep.from_host(sp, dev)
    buf2 = S.StepBuffers.make(kv, d2, msl, dev)
    slots = []
    for ds, bs in ((d, buf), (d2, buf2)):
        oh = [torch.empty(bs.accept.shape, dtype=torch.int32).pin_memory(),
              torch.empty(bs.out_tok.shape, dtype=torch.int32).pin_memory(),
              torch.empty(bs.num_out.shape, dtype=torch.int32).pin_memory()]
        slots.append((ds, bs, oh, torch.cuda.Event(), torch.cuda.Event()))  # copied, inputs free
    d2h = sum(t.numel() * 4 for t in slots[0][2])
    cs = torch.cuda.Stream(dev)

    def step_e2e(i):
        ds, bs, oh, copied, free = slots[i % 2]
        if i >= 2:
            cs.wait_event(free)  # step i - 2 has finished reading this slot's inputs
        with torch.cuda.stream(cs):
            for k in names:
                getattr(ds, k).copy_(host[k], non_blocking=True)
        copied.record(cs)
        stream.wait_event(copied)
        S.run_step(kv, ds, bs, msl, stream)
        free.record(stream)
        oh[0].copy_(bs.accept, non_blocking=True)
        oh[1].copy_(bs.out_tok, non_blocking=True)
        oh[2].copy_(bs.num_out, non_blocking=True)

    for i in range(max(3, args.warmup)):
        step_e2e(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(10, args.steps // 2)
    torch.cuda.synchronize()
    a.record(stream)
    cs.wait_event(a)
    for i in range(n):
        step_e2e(i)
    b.record(stream)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0 and int(buf2.status.item()) == 0, "device status set in the end-to-end steps"
    ms = a.elapsed_time(b)
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return {"value": d.batch * n * world / (ms / 1e3), "unit": "seqs/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": ms / n, "steps": n,
            "pipeline": "two input buffers: step i + 1's H2D on a second stream overlaps step i's kernels"}


# ----------------------------------------------------------------------------
# reference arm: the CPU oracle
# ----------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    case, desc = make_case(args.config, args.temperature, args.steps + args.warmup + 2)
    cores = oracle.set_threads(os.cpu_count() or 1)  # the oracle's OpenMP tasks on every host core
    n, t1 = cpu_seqs_for(case, budget_s=0.5)
    seqs = list(range(n))
    for _ in range(args.warmup):
        oracle_sample_step(case, seqs)
    ts = [oracle_sample_step(case, seqs) for _ in range(args.steps)]
    total = float(np.sum(ts))
    value = n * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "seqs/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded numpy PCG64; no dataset or weights)",
        "config": {"workload": desc, "global_batch": case.state.batch},
        "cpu_baseline": {"value": value, "unit": "seqs/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: the oracle's verify step for {n} of the {case.state.batch} "
                                   f"sequences (fp64 C, OpenMP on {cores} threads)"},
        "e2e": {"value": value, "unit": "seqs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
