"""Benchmark of the DSpark draft-and-verify step on GB300.

One step = the whole hot path on one block of the full-geometry drafter at
bs=1, ctx 4096 (seeded synthetic inputs, bf16 weights): fc context fusion, 5
MLA block-diffusion layers + lm_head, Markov rollout, confidence head, greedy
verification. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the float64 CPU oracle on the host cores on a bounded
sample of the same workload (the method has no other reference implementation).
Multi-GPU: replicas only (every rank runs its own step; no data-path collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# --oracle-threads N: the oracle's BLAS threads must be fixed before numpy loads
for _i, _a in enumerate(sys.argv):
    if _a.startswith("--oracle-threads"):
        _n = _a.split("=", 1)[1] if "=" in _a else (sys.argv[_i + 1] if _i + 1 < len(sys.argv) else "0")
        if _n.isdigit() and int(_n) > 0:
            for _k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
                os.environ[_k] = _n

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "µs per 7-token draft block at bs=1 (full geometry); achieved HBM TB/s vs peak"
UNIT = "us"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


def gemm_kernel_name(fmt: str, M: int) -> str:
    """The weight-GEMM kernel the library launches for this format at M activation rows."""
    bn = min(224, max(16, 1 << (M - 1).bit_length()))
    if fmt == "bf16":
        return f"gemm_swapab_kernel<{bn}>"
    if fmt == "fp8" and bn <= 32:
        return f"gemm_f8_kernel<{8 if M <= 8 else bn}>"
    return f"gemm_q_kernel<{bn}, {fmt}>"


def algorithmic_bytes(G, ctx, bs: int = 1, fmt: str = "bf16"):
    """Bytes one step must move at least: every weight once (w2 once, the
    block's 7 rows of w1), fp32 gains and confidence head, the latent KV once,
    the aux states, z and ell written once and read once, the target logits.
    FP8 / NVFP4 (fc, q_b, o, gate, up, down): 1 byte + a 4-byte scale per row, or
    half a byte + one scale byte per 16."""
    lp = G.layer_params()
    mats = sum(v for k, v in lp.items() if k != "norms")
    c = G.param_counts()
    qn = c["quantised"]
    q_rows = G.hidden + G.n_layers * (G.n_heads * G.q_head_dim + G.hidden + 2 * G.inter + G.hidden)
    per = {"bf16": 2.0, "fp8": 1.0, "nvfp4": 0.5 + 1.0 / 16, "mxfp4": 0.5 + 1.0 / 32}[fmt]
    extra = {"bf16": 0, "fp8": 4 * q_rows, "nvfp4": 0, "mxfp4": 0}[fmt]
    w_bf16 = 2 * (c["fc"] + G.n_layers * mats + c["lm_head"] + G.rank * G.vocab + bs * G.block * G.rank) \
        - int(2 * qn) + int(per * qn) + extra
    w_f32 = 4 * (G.n_layers * lp["norms"] + 2 * G.hidden)
    ctx_total = sum(ctx) if isinstance(ctx, (list, tuple)) else bs * ctx
    kv = G.n_layers * ctx_total * G.kv_dim * 2
    aux = bs * G.block * G.n_aux * G.hidden * 2
    logits = 4 * bs * G.vocab * (2 * G.block + 2 * G.block + (G.block + 1))
    total = w_bf16 + w_f32 + kv + aux + logits
    return {"weights": w_bf16 + w_f32, "kv": kv, "aux": aux, "logits": logits, "total": total,
            "fc_weight": int(per * c["fc"]) + (4 * G.hidden if fmt == "fp8" else 0)}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_figures(ms_step: float, e2e_ms_step: float, world: int, bs: int, block: int) -> dict:
    """Whole-job figures of N replicas from the per-step times (already the
    maximum over ranks): every rank drafts bs blocks per step at once, so the job
    spends ms_step / N per block and drafts block * bs * N tokens per step."""
    return {"us_per_block": ms_step * 1e3 / world, "e2e_us_per_block": e2e_ms_step * 1e3 / world,
            "drafted_tokens_per_s": block * bs * world / (ms_step * 1e-3)}


def run_config(w, ctx_list, world: int, draft_mode: int, verify_mode: int, T: float, top_p: float, fmt: str,
               total_bytes: int) -> dict:
    """The JSON line's config: the workload and its replicas."""
    G, bs = w.geom, w.bs
    max_ctx = max(ctx_list)
    return {"workload": w.name, "model": "DSpark drafter (Kimi-K3 geometry), random init",
            "global_batch": bs * world, "blocks_per_step": bs * world,
            "seq_len": max_ctx if bs == 1 else f"{min(ctx_list)}..{max_ctx} (mean {statistics.mean(ctx_list):.0f})",
            "block": G.block, "draft": MODE_NAMES[draft_mode], "verify": MODE_NAMES[verify_mode],
            "temperature": T if (draft_mode or verify_mode) else None,
            "top_p": top_p if (draft_mode or verify_mode) else None, "weights": fmt,
            "rope": "yarn-16 from 65536" if G.yarn_factor > 1 else "plain",
            "parallelism": f"replicas{world}",
            "l2": f"no flush: working set {total_bytes / 1e9:.2f} GB per step > 129 MB L2"}


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm): one whole block, float64
# ---------------------------------------------------------------------------
LAYER_KEYS = ("attn_norm", "w_qkv_a", "q_a_norm", "kv_a_norm", "w_q_b", "w_kv_b", "w_o", "mlp_norm", "w_gate", "w_up",
              "w_down")


def _mem_available_bytes() -> int:
    """Host memory this process may still use: MemAvailable, capped by a cgroup limit."""
    avail = 0
    try:
        with open("/proc/meminfo") as f:
            for ln in f:
                if ln.startswith("MemAvailable:"):
                    avail = int(ln.split()[1]) * 1024
    except OSError:
        pass
    for cg in ("/sys/fs/cgroup/memory.max", "/sys/fs/cgroup/memory/memory.limit_in_bytes"):
        try:
            with open(cg) as f:
                v = f.read().strip()
            if v.isdigit():
                avail = min(avail, int(v)) if avail else int(v)
        except OSError:
            pass
    return avail


class OracleWeights:
    """float64 copies of the drafter's weights for the oracle (input preparation: the
    bf16 -> float64 conversion is exact). Kept across blocks when the host has room
    for them (about 8 bytes per parameter), else converted again at every use. The
    conversion time is reported apart from the oracle's compute time."""

    LM_CHUNK = 8192

    def __init__(self, W, G):
        self.W, self.G = W, G
        need = 8 * sum(int(t.numel()) for t in W.values() if torch.is_tensor(t))
        self.keep = _mem_available_bytes() > 3 * need
        self.cache = {}
        self.conv_s = 0.0

    def get(self, name, lo=None, hi=None):
        key = (name, lo, hi)
        if key in self.cache:
            return self.cache[key]
        t0 = time.perf_counter()
        t = self.W[name] if lo is None else self.W[name][lo:hi]
        a = t.detach().to(torch.float64).cpu().numpy()
        self.conv_s += time.perf_counter() - t0
        if self.keep:
            self.cache[key] = a
        return a

    def lm_chunks(self):
        V = self.G.vocab
        for lo in range(0, V, self.LM_CHUNK):
            yield lo, self.get("w_lm", lo, min(V, lo + self.LM_CHUNK))


def oracle_block(OW, G, I, b, draft_mode, verify_mode, T, top_p, P=None):
    """One whole block of the float64 oracle for sequence b: fc fusion, every layer,
    the final norm, the full lm_head, the Markov rollout, the confidence head and the
    verification the workload uses (greedy, token-wise probabilistic or block).
    Returns the seconds of oracle compute; weight conversions are not counted
    (OW.conv_s holds them)."""
    from oracle import network as N
    from oracle import sampling as S
    ctx = I["ctx_list"][b]
    conv0 = OW.conv_s
    f64 = lambda t: t.detach().to(torch.float64).cpu().numpy()
    aux = f64(I["aux"][b])
    table = I["page_table"][b]
    pages = table[: (ctx + G.page_size - 1) // G.page_size].long()
    caches = []
    for l in range(G.n_layers):
        pool = f64(I["kv_pools"][l][pages])
        caches.append(N.gather_cache(pool, np.arange(pool.shape[0]), ctx))
    w1, w2 = OW.W["markov_w1"].cpu(), OW.W["markov_w2"].cpu()
    t0 = time.perf_counter()
    x = N.fuse_ctx(OW.get("w_fc"), aux)
    pos = np.arange(G.block, dtype=np.float64) + ctx
    for l in range(G.n_layers):
        L = {k: OW.get(f"l{l}.{k}") for k in LAYER_KEYS}
        x = N.layer(x, L, G, caches[l][:, :G.kv_lora], caches[l][:, G.kv_lora:], pos)
    h = N.rmsnorm(x, OW.get("final_norm"), G.eps)
    z = np.empty((G.block, G.vocab), dtype=np.float64)
    for lo, wl in OW.lm_chunks():
        z[:, lo:lo + wl.shape[0]] = h @ wl.T
    zf = z.astype(np.float32)
    anchor = int(I["anchor"][b])
    toks, ell = S.markov_rollout(zf, w1, w2, anchor, draft_mode, T, top_p, seed=1, seq=b, step=0)
    N.confidence(h, OW.get("w_conf"), float(OW.W["b_conf"].item()))
    Pb = np.concatenate([ell, ell[-1:]]).astype(np.float32) if P is None else P
    if verify_mode == 0:
        S.verify_greedy(Pb, toks)
    elif verify_mode == 1:
        S.verify_prob(Pb, ell, toks, draft_mode, T, top_p, seed=1, seq=b, step=0)
    else:
        S.verify_block(Pb, ell, toks, draft_mode, T, top_p, seed=1, seq=b, step=0)
    t1 = time.perf_counter()
    return (t1 - t0) - (OW.conv_s - conv0)


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def oracle_threads() -> int:
    """Threads the oracle's BLAS may use (the --oracle-threads setting, else every core)."""
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        v = os.environ.get(k)
        if v and v.isdigit():
            return int(v)
    return cores()


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------
def select_workload(args):
    """The workload of one bench line and its sampling modes: (workload, draft, verify, T, top_p)."""
    from synthetic.configs import BATCH_STEP, FP8_STEP, FULL_STEP, LONG_STEP, MXFP4_STEP, NVFP4_STEP
    if args.workload == "full_bs1_ctx4096":
        w = {"bf16": FULL_STEP, "fp8": FP8_STEP, "nvfp4": NVFP4_STEP, "mxfp4": MXFP4_STEP}[args.format]
    else:
        if args.format != "bf16":
            raise SystemExit("--format applies to the full_bs1_ctx4096 workload")
        w = {"full_bs1_ctx95000_yarn": LONG_STEP, "full_bs32_paged": BATCH_STEP}[args.workload]
    draft, verify, T, top_p = w.draft_mode, w.verify_mode, w.temperature, w.top_p
    if args.sampling == "probabilistic":  # the cards' production sampling: T 1.0, top_p 0.95
        draft, verify, T, top_p = 1, 1, 1.0, 0.95
    elif args.sampling == "greedy":
        draft, verify = 0, 0
    if args.verify == "block":
        verify = 2
        if draft == 0 and args.sampling is None:
            T, top_p = 1.0, 0.95
    elif args.verify == "probabilistic":
        verify = 1
        if draft == 0 and args.sampling is None:
            T, top_p = 1.0, 0.95
    return w, draft, verify, T, top_p


MODE_NAMES = {0: "greedy", 1: "probabilistic", 2: "block"}


def attention_flops(G, ctx_list, with_block: bool = True) -> float:
    """Tensor-core attention FLOPs of one step: every query row of every head against
    every key (scores over the 576-wide key, P V over the 512-wide latent)."""
    R = G.block * G.n_heads
    keys = sum(c + (G.block if with_block else 0) for c in ctx_list)
    return 2.0 * R * keys * (G.kv_lora + G.d_rope + G.kv_lora) * G.n_layers


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="full_bs1_ctx4096",
                    choices=["full_bs1_ctx4096", "full_bs1_ctx95000_yarn", "full_bs32_paged"],
                    help="full_bs1_ctx4096: the headline (bs 1, ctx 4096); full_bs1_ctx95000_yarn: 95,000-token "
                         "latent cache, YaRN-16, probabilistic draft and verify at T 1.0, top_p 0.95; "
                         "full_bs32_paged: 32 sequences, paged ragged contexts in [1k, 16k], greedy")
    ap.add_argument("--sampling", choices=["greedy", "probabilistic"], default=None,
                    help="draft and verify sampling (default: the workload's); probabilistic = T 1.0, top_p 0.95")
    ap.add_argument("--verify", choices=["greedy", "probabilistic", "block"], default=None,
                    help="verification rule (default: the workload's)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-threads", type=int, default=0,
                    help="threads of the oracle's BLAS (set before numpy loads; 0: every core)")
    ap.add_argument("--only", choices=["fc", "rollout", "layer", "append", "verify"], default=None,
                    help="time one call alone for profiling: fc (the fusion GEMM; full shape unless --fc-hidden), "
                         "rollout (Markov rollout, full vocabulary), layer (one full-width MLA layer, ctx 4096), "
                         "append (latent-cache append of 8 verified tokens, all 5 layers, full hidden/latent)")
    ap.add_argument("--fc-hidden", type=int, default=0, help="--only fc: hidden size (output channels)")
    ap.add_argument("--fc-aux", type=int, default=0, help="--only fc: captured states (K = aux * hidden)")
    ap.add_argument("--roll-mode", choices=["greedy", "probabilistic"], default="greedy",
                    help="--only rollout: draft sampling (probabilistic: T 1.0, top_p 0.95)")
    ap.add_argument("--roll-bs", type=int, default=1, help="--only rollout: sequences per call (1..32)")
    ap.add_argument("--format", choices=["bf16", "fp8", "nvfp4", "mxfp4"], default="bf16",
                    help="weight format of fc, q_b, o, gate, up, down (the weight-format sweep workloads)")
    ap.add_argument("--no-drift", action="store_true", help="--format fp8|nvfp4|mxfp4: skip the drift report")
    ap.add_argument("--drift", action="store_true",
                    help="run the weight-format drift / acceptance-ceiling harness instead of the step benchmark")
    ap.add_argument("--blocks", type=int, default=1024, help="--drift: blocks per aux regime")
    ap.add_argument("--regime", choices=["boot", "heavy", "gauss", "all"], default="all", help="--drift: aux regime")
    ap.add_argument("--drift-formats", default="fp8,nvfp4,mxfp4", help="--drift: formats against the bf16 path")
    ap.add_argument("--drift-geom", choices=["full", "mid"], default="full",
                    help="--drift: full drafter geometry, or a small one for a quick check")
    ap.add_argument("--drift-oracle-blocks", type=int, default=0,
                    help="--drift: also compare bf16 and every format with the float64 oracle on this many blocks "
                         "per regime (the FP32-reference rows)")
    args = ap.parse_args()
    if args.drift:
        return drift_harness(args)
    assert args.warmup >= 3 or args.impl == "reference", "at least 3 warm-up steps"

    from synthetic import generate as gen
    w, draft_mode, verify_mode, T, top_p = select_workload(args)
    G = w.geom
    world, rank, local = dist_setup()
    ctx_list = gen.context_lengths(w)
    max_ctx = max(ctx_list)
    bs = w.bs
    ab = algorithmic_bytes(G, ctx_list, bs=bs, fmt=args.format)
    config = run_config(w, ctx_list, world, draft_mode, verify_mode, T, top_p, args.format, ab["total"])

    if args.only == "fc":
        return only_fc(args, G, world, rank, local)
    if args.only == "append":
        return only_append(args, G, local)
    if args.only == "verify":
        return only_verify(args, G, local)
    if args.only in ("rollout", "layer"):
        return only_call(args, G, local)

    if args.impl == "reference":
        if rank != 0:
            return
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        W = gen.make_weights(w, dev)
        I = gen.make_inputs(w, dev)
        from oracle import build as obuild
        obuild.build()
        OW = OracleWeights(W, G)
        for _ in range(args.warmup):
            oracle_block(OW, G, I, 0, draft_mode, verify_mode, T, top_p)
        vals = []
        for k in range(args.steps):
            vals.append(oracle_block(OW, G, I, 0, draft_mode, verify_mode, T, top_p) * bs * 1e6)
        v = statistics.median(vals)
        sample = (f"per step: one whole block of sequence 0 ({G.n_layers} layers, ctx {ctx_list[0]}, the full "
                  f"lm_head, rollout, confidence, {MODE_NAMES[verify_mode]} verify), float64"
                  + (f", times {bs} sequences" if bs > 1 else ""))
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": v / 1e3, "higher_is_better": False, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": v, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
                                 "sample": sample, "weight_conversion_s": round(OW.conv_s, 1),
                                 "weights_kept": OW.keep},
                "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import mla_block_diffusion_gb300 as M
    from mla_block_diffusion_gb300 import build as libbuild
    from oracle import build as obuild
    libbuild.build()
    obuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    W = gen.make_weights(w, dev)
    I = gen.make_inputs(w, dev)
    Wd = W
    if args.format != "bf16":
        from synthetic import quantize as Q
        Wd = Q.quantise_weights(W, args.format, G.n_layers)
        torch.cuda.empty_cache()
    ds = M.DSpark(G, Wd, max_bs=bs, max_ctx=max_ctx, weight_format=w.weight_format)
    kv = ds.make_kv(I["kv_pools"], I["page_table"], I["ctx_len"], max_ctx)
    x = torch.empty(bs, G.block, G.hidden, dtype=torch.float32, device=dev)
    h_out = torch.empty_like(x)
    z = torch.empty(bs, G.block, G.vocab, dtype=torch.float32, device=dev)
    ell = torch.empty_like(z)
    tokens = torch.empty(bs, G.block, dtype=torch.int32, device=dev)
    conf = torch.empty(bs, G.block, dtype=torch.float32, device=dev)
    acc = torch.empty(bs, dtype=torch.int32, device=dev)
    out = torch.empty(bs, G.block + 1, dtype=torch.int32, device=dev)
    P = torch.empty(bs, G.block + 1, G.vocab, dtype=torch.float32, device=dev)
    smp = M.Sample(draft_mode, verify_mode, T, top_p, 1, 0)
    aux, anchor = I["aux"], I["anchor"]

    def step():
        ds.fuse_ctx(aux, x, bs)
        ds.draft_block(x, kv, h_out, z, bs)
        ds.markov_rollout(z, anchor, smp, tokens, ell, bs)
        ds.confidence(h_out, conf, bs)
        ds.verify(P, ell, tokens, smp, acc, out, bs)

    # the target's logits: the drafter's own Markov logits plus N(0, sigma^2) noise,
    # fixed from the first pass (the step is deterministic, so they match every step)
    P.zero_()
    step()
    st = ds.check()
    assert st == 0, f"device error {st}"
    noise = gen.noise((bs, G.block + 1, G.vocab), w.target_noise, w.input_seed, device=dev)
    P.copy_(torch.cat([ell, ell[:, -1:]], dim=1) + noise)
    del noise
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert ds.check() == 0

    # ---- the whole step as one CUDA graph (eager launches if capture is refused) ----
    graph = None
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        g.replay()
        torch.cuda.synchronize()
        if ds.check() == 0:
            graph = g
    except Exception as e:  # noqa: BLE001
        torch.cuda.synchronize()
        ds.check()
        config["graph_error"] = str(e)[:200]
    run = graph.replay if graph is not None else step
    config["launch"] = "cuda_graph" if graph is not None else "eager"
    for _ in range(3):
        run()

    # ---- device-resident timing ----
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    start.record()
    for k in range(args.steps):
        run()
    stop.record()
    torch.cuda.synchronize()
    barrier(world)
    clocks = clk.stop()
    assert ds.check() == 0
    ms = start.elapsed_time(stop) / args.steps
    ms = max_over_ranks(ms, world)

    def timed(call, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize()
        for a_, b_ in evs:
            a_.record()
            call()
            b_.record()
        torch.cuda.synchronize()
        return statistics.mean(a_.elapsed_time(b_) for a_, b_ in evs)

    pk, src = peaks()
    hbm = pk["hbm_gbs"]
    roofline = None
    if G.yarn_factor > 1 or max_ctx > 32768:
        # long context: the attention is the dominant kernel and tensor-bound. Its
        # KV-dependent time is the difference between the layers at the workload's
        # context and the same launches with every context length set to 0 (same
        # grid: the splits beyond the context exit at once).
        zero_ctx = torch.zeros_like(I["ctx_len"])
        kv0 = ds.make_kv(I["kv_pools"], I["page_table"], zero_ctx, max_ctx)
        n = max(3, args.steps // 2)
        ms_ctx = timed(lambda: (ds.fuse_ctx(aux, x, bs), ds.draft_block(x, kv, h_out, z, bs)), n)
        ms_0 = timed(lambda: (ds.fuse_ctx(aux, x, bs), ds.draft_block(x, kv0, h_out, z, bs)), n)
        fl = attention_flops(G, ctx_list, with_block=False)
        tf_peak = pk.get("bf16_tflops_sustained", pk.get("bf16_tflops", FALLBACK["bf16_tflops"]))
        d = max(ms_ctx - ms_0, 1e-6)
        achieved = fl / (d * 1e-3) / 1e12
        roofline = {"kernel": "mla_attention_tc_kernel<576,512> (KV part, all layers: draft layers at the context "
                              "minus the same launches at context 0)",
                    "bound": "tensor", "achieved": achieved, "peak": tf_peak, "unit": "TFLOP/s",
                    "frac": achieved / tf_peak, "traffic": None, "algorithmic_flops_per_step": fl,
                    "kv_part_ms": d, "draft_ms_at_ctx": ms_ctx, "draft_ms_at_ctx0": ms_0,
                    "peak_source": src + " (sustained bf16)"}
    # ---- the GEMM (dominant kernel class at short context): the fc fusion launch, which
    # the API isolates (the same gemm_swapab_kernel as the step's other 26 weight GEMMs;
    # 514 MB of weights > L2) ----
    fc_ms = timed(lambda: ds.fuse_ctx(aux, x, bs), args.steps)
    fc_bytes = ab["fc_weight"] + bs * G.block * G.n_aux * G.hidden * 2 + bs * G.block * G.hidden * 4
    fc_achieved = fc_bytes / (fc_ms * 1e-3) / 1e9
    traffic = None
    # ncu DRAM bytes of this launch, valid while the kernel's source is the profiled one
    tsrc = {"bf16": ("fc_gemm_traffic.json", "gemm.cuh", "gemm_cuh_sha256"),
            "fp8": ("fc_gemm_f8_traffic.json", "gemm_f8.cuh", "gemm_f8_cuh_sha256")}.get(args.format)
    if tsrc and bs == 1 and os.path.exists(os.path.join(ROOT, "profiles", tsrc[0])):
        with open(os.path.join(ROOT, "profiles", tsrc[0])) as f:
            td = json.load(f)
        h = hashlib.sha256(open(os.path.join(ROOT, "mla_block_diffusion_gb300", "csrc", tsrc[1]), "rb").read())
        if td.get(tsrc[2]) == h.hexdigest():
            traffic = td.get("dram_bytes_per_launch")
    gemm_line = {"kernel": gemm_kernel_name(args.format, bs * G.block) + " (fc fusion launch; the step's "
                                                                         "weight-GEMM class)",
                 "bound": "hbm", "achieved": fc_achieved, "peak": hbm, "unit": "GB/s", "frac": fc_achieved / hbm,
                 "traffic": traffic, "algorithmic_bytes_per_launch": fc_bytes, "avg_launch_ms": fc_ms,
                 "peak_source": src,
                 "why_this_launch": ("the weight GEMMs are one kernel class (27 launches per step, about three "
                                     "quarters of the serialised step; the lm_head the longest launch at about "
                                     "355 us for 2.35 GB); the fc fusion is the one launch of that class the API "
                                     "isolates (dspark_fuse_ctx), with the same kernel and tiles as the lm_head "
                                     "and 514 MB of weights, larger than L2, so CUDA events time it alone; the "
                                     "class's launches and shares: profiles/step_launches_*.md")
                 if args.format == "bf16" else
                 ("the fc fusion is the one launch of the quantised GEMM kernel (21 launches per step: fc, q_b, o, "
                  "gate/up, down) that the API isolates (dspark_fuse_ctx); q_a||kv_a and the lm_head stay bf16; "
                  "the launches and shares: profiles/step_launches_*.md")}
    if roofline is None:
        roofline = gemm_line
    else:
        roofline["gemm"] = gemm_line

    # ---- end to end through the public API with host buffers ----
    aux_h = aux.cpu().pin_memory()
    anchor_h = anchor.cpu().pin_memory()
    P_h = P.cpu().pin_memory()
    acc_h = torch.empty_like(acc, device="cpu").pin_memory()
    out_h = torch.empty_like(out, device="cpu").pin_memory()
    conf_h = torch.empty_like(conf, device="cpu").pin_memory()
    tok_h = torch.empty_like(tokens, device="cpu").pin_memory()

    def e2e_step():
        aux.copy_(aux_h, non_blocking=True)
        anchor.copy_(anchor_h, non_blocking=True)
        P.copy_(P_h, non_blocking=True)
        run()
        acc_h.copy_(acc, non_blocking=True)
        out_h.copy_(out, non_blocking=True)
        conf_h.copy_(conf, non_blocking=True)
        tok_h.copy_(tokens, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(2):
        e2e_step()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / args.steps, world)
    h2d = aux_h.numel() * aux_h.element_size() + anchor_h.numel() * 4 + P_h.numel() * 4
    d2h = (acc_h.numel() + out_h.numel() + tok_h.numel()) * 4 + conf_h.numel() * 4
    accept = acc.cpu().tolist()

    gpu_launches_per_step = ds_launches_per_step(ds, bs=bs, draft_mode=draft_mode, verify_mode=verify_mode)
    jf = job_figures(ms, e2e_ms, world, bs, G.block)  # whole job: every rank runs its own step
    line = {
        "metric": METRIC, "value": jf["us_per_block"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic", "config": config,
        "drafted_tokens_per_s": jf["drafted_tokens_per_s"],
        "hbm": {"algorithmic_bytes_per_step": ab["total"], "achieved_TBps": ab["total"] / (ms * 1e-3) / 1e12,
                "frac_of_peak": ab["total"] / (ms * 1e-3) / 1e9 / hbm, "peak_GBps": hbm, "peak_source": src,
                "frac_of_8TBps": ab["total"] / (ms * 1e-3) / 8e12},
        "roofline": roofline,
        "clocks": clocks,
        "e2e": {"value": jf["e2e_us_per_block"], "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": gpu_launches_per_step * args.steps,
        "accept_len": accept if bs <= 8 else {"histogram_0_to_7": np.bincount(np.asarray(accept), minlength=G.block + 1)
                                                                     .tolist()},
    }
    if G.yarn_factor > 1 or max_ctx > 32768:
        line["attention_flops_per_step"] = attention_flops(G, ctx_list)
    if args.format != "bf16" and not args.no_drift and rank == 0:
        line["drift"] = drift_report(w, W, I, h_out, z, max_ctx)
        line["vs_bf16_note"] = "drift: this format's GPU outputs against the float64 oracle on the original bf16 weights"
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        OW = OracleWeights(W, G)
        secs = oracle_block(OW, G, I, 0, draft_mode, verify_mode, T, top_p,
                            P=P[0].cpu().numpy() if bs == 1 else None)
        line["cpu_baseline"] = {"value": secs * bs * 1e6, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
                                "sample": f"one whole block of sequence 0 ({G.n_layers} layers, ctx {ctx_list[0]}, the "
                                          f"full lm_head, rollout, confidence, {MODE_NAMES[verify_mode]} verify), "
                                          f"float64" + (f", times {bs} sequences" if bs > 1 else "")
                                          + f"; weight conversion {OW.conv_s:.1f} s not counted"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def drift_report(w, W, I, h_out, z, ctx):
    """Weight-format drift: the GPU outputs with quantised weights against the
    float64 oracle on the original bf16 weights (hidden-state relative error, logit
    relative error, per-position greedy agreement)."""
    from oracle import network as N
    G = w.geom
    f64 = lambda t: t.detach().to(torch.float64).cpu().numpy()
    keys = ["attn_norm", "w_qkv_a", "q_a_norm", "kv_a_norm", "w_q_b", "w_kv_b", "w_o", "mlp_norm", "w_gate", "w_up",
            "w_down"]
    x = N.fuse_ctx(f64(W["w_fc"]), f64(I["aux"][0]))
    table = I["page_table"][0]
    pages = table[: (ctx + G.page_size - 1) // G.page_size].long()
    pos = np.arange(G.block, dtype=np.float64) + ctx
    for l in range(G.n_layers):
        L = {k: f64(W[f"l{l}.{k}"]) for k in keys}
        pool = f64(I["kv_pools"][l][pages])
        cache = N.gather_cache(pool, np.arange(pool.shape[0]), ctx)
        x = N.layer(x, L, G, cache[:, :G.kv_lora], cache[:, G.kv_lora:], pos)
    h = N.rmsnorm(x, f64(W["final_norm"]), G.eps)
    zo = np.empty((G.block, G.vocab))
    for lo in range(0, G.vocab, 16384):
        zo[:, lo:lo + 16384] = h @ f64(W["w_lm"][lo:lo + 16384]).T
    hg, zg = h_out[0].double().cpu().numpy(), z[0].double().cpu().numpy()
    rel = lambda a, b: float(np.linalg.norm(a - b) / np.linalg.norm(b))
    agree = float(np.mean(np.argmax(zg, axis=1) == np.argmax(zo, axis=1)))
    return {"h_out_rel_l2": rel(hg, h), "z_rel_l2": rel(zg, zo), "greedy_agreement": agree}


def only_fc(args, G, world, rank, local):
    """The fc fusion GEMM alone at its full shape: 7168 x 35840 bf16 weights (514 MB, > L2),
    7 rows; the rest of the drafter is shrunk so the device holds well under 1 GB."""
    from dataclasses import replace
    import mla_block_diffusion_gb300 as M
    from mla_block_diffusion_gb300 import build as libbuild
    from synthetic import generate as gen
    from synthetic.configs import FULL_STEP
    libbuild.build()
    torch.cuda.set_device(local)
    g = replace(G, n_layers=1, n_heads=4, q_lora=64, kv_lora=64, d_nope=32, d_rope=16, d_v=16, inter=64, vocab=128,
                rank=16)
    if args.fc_hidden:
        g = replace(g, hidden=args.fc_hidden, n_aux=args.fc_aux or G.n_aux)
    w = replace(FULL_STEP, geom=g)
    W = gen.make_weights(w, "cuda")
    aux = gen.make_inputs(w, "cuda")["aux"]
    fmt = args.format
    if fmt != "bf16":  # the weight-only formats need every quantised dimension aligned
        from synthetic import quantize as Q
        from synthetic.configs import FORMAT_FP8, FORMAT_MXFP4, FORMAT_NVFP4
        g = replace(g, q_lora=512, d_v=128, inter=512)
        w = replace(FULL_STEP, geom=g)
        W = Q.quantise_weights(gen.make_weights(w, "cuda"), fmt, g.n_layers)
        ds = M.DSpark(g, W, max_bs=1,
                      weight_format={"fp8": FORMAT_FP8, "nvfp4": FORMAT_NVFP4, "mxfp4": FORMAT_MXFP4}[fmt])
    else:
        ds = M.DSpark(g, W, max_bs=1)
    x = torch.empty(1, g.block, g.hidden, dtype=torch.float32, device="cuda")
    for _ in range(args.warmup):
        ds.fuse_ctx(aux, x, 1)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for a_, b_ in evs:
        a_.record()
        ds.fuse_ctx(aux, x, 1)
        b_.record()
    torch.cuda.synchronize()
    assert ds.check() == 0
    ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in evs)
    per = {"bf16": 2.0, "fp8": 1.0, "nvfp4": 0.5 + 1.0 / 16, "mxfp4": 0.5 + 1.0 / 32}[fmt]
    nbytes = int(per * g.hidden * g.n_aux * g.hidden) + g.block * g.n_aux * g.hidden * 2 + g.block * g.hidden * 4
    pk, src = peaks()
    if rank == 0:
        kern = gemm_kernel_name(fmt, g.block)
        print(json.dumps({"kernel": f"{kern} fc fusion", "format": fmt, "avg_launch_ms": ms,
                          "algorithmic_bytes_per_launch": nbytes, "achieved_GBps": nbytes / (ms * 1e-3) / 1e9,
                          "peak_GBps": pk["hbm_gbs"], "peak_source": src}))


def only_call(args, G, local):
    """One API call alone on a drafter shrunk everywhere else (for ncu captures):
    rollout: full vocabulary and rank (w1, w2 84 MB each), greedy;
    layer: one layer of full attention width (64 heads, latent 512 + 64) at ctx 4096."""
    from dataclasses import replace
    import mla_block_diffusion_gb300 as M
    from mla_block_diffusion_gb300 import build as libbuild
    from synthetic import generate as gen
    from synthetic.configs import FULL_STEP
    libbuild.build()
    torch.cuda.set_device(local)
    if args.only == "rollout":
        g = replace(G, hidden=64, n_aux=1, n_layers=1, n_heads=1, q_lora=64, kv_lora=64, d_nope=16, d_rope=16, d_v=64,
                    inter=64)
    else:
        g = replace(G, hidden=1024, n_aux=1, n_layers=1, q_lora=256, inter=64, vocab=128, rank=16)
    w = replace(FULL_STEP, geom=g)
    W = gen.make_weights(w, "cuda")
    I = gen.make_inputs(w, "cuda")
    ctx = I["ctx_list"][0]
    rbs = args.roll_bs if args.only == "rollout" else 1
    ds = M.DSpark(g, W, max_bs=rbs, max_ctx=ctx)
    x = torch.empty(1, g.block, g.hidden, dtype=torch.float32, device="cuda")
    h = torch.empty_like(x)
    z = gen.draft_logits(rbs, g.block, g.vocab, 1, device="cuda")
    ell = torch.empty_like(z)
    tokens = torch.empty(rbs, g.block, dtype=torch.int32, device="cuda")
    gen_a = torch.Generator().manual_seed(7)
    anchors = torch.randint(0, g.vocab, (rbs,), generator=gen_a, dtype=torch.int32).cuda() if rbs > 1 else I["anchor"]
    kv = ds.make_kv(I["kv_pools"], I["page_table"], I["ctx_len"], ctx)
    prob = args.only == "rollout" and args.roll_mode == "probabilistic"
    smp = M.Sample(M.PROBABILISTIC, M.PROBABILISTIC, 1.0, 0.95, 1, 0) if prob else M.Sample(M.GREEDY, M.GREEDY, 1.0,
                                                                                             1.0, 1, 0)

    def call():
        if args.only == "rollout":
            ds.markov_rollout(z, anchors, smp, tokens, ell, rbs)
        else:
            ds.fuse_ctx(I["aux"], x, 1)
            ds.draft_block(x, kv, h, z, 1)

    for _ in range(args.warmup):
        call()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for a_, b_ in evs:
        a_.record()
        call()
        b_.record()
    torch.cuda.synchronize()
    assert ds.check() == 0
    print(json.dumps({"only": args.only, "bs": rbs, "avg_call_ms": statistics.mean(a_.elapsed_time(b_) for a_, b_ in evs)}))


def only_append(args, G, local):
    """dspark_kv_append alone: 8 newly verified tokens of one sequence into all layers' page pools,
    full hidden size and latent width (the other dimensions shrunk; the device holds < 1 GB).
    Algorithmic bytes: the kv_a rows of every layer's fused q_a || kv_a weights, the context
    features and the written entries."""
    from dataclasses import replace
    import mla_block_diffusion_gb300 as M
    from mla_block_diffusion_gb300 import build as libbuild
    from synthetic import generate as gen
    from synthetic.configs import FULL_STEP
    libbuild.build()
    torch.cuda.set_device(local)
    g = replace(G, inter=64, vocab=128, rank=16)
    w = replace(FULL_STEP, geom=g)
    W = gen.make_weights(w, "cuda")
    I = gen.make_inputs(w, "cuda")
    ctx0 = I["ctx_list"][0]
    n = g.block + 1
    P = g.page_size
    # one spare page after the sequence's pages
    table = torch.cat([I["page_table"], torch.full((1, 1), I["n_pages"], dtype=torch.int32, device="cuda")], dim=1)
    pools = [torch.cat([p, torch.zeros((1, P, g.kv_dim), dtype=p.dtype, device="cuda")]) for p in I["kv_pools"]]
    ctx = torch.tensor([ctx0], dtype=torch.int32, device="cuda")
    ds = M.DSpark(g, W, max_bs=1, max_ctx=ctx0 + n)
    kv = ds.make_kv(pools, table, ctx, ctx0 + n)
    x_new = gen.normal((1, n, g.hidden), 1.0, 7, "x_new", "cuda").float()
    n_new = torch.tensor([n], dtype=torch.int32, device="cuda")
    times = []
    for k in range(args.warmup + args.steps):
        ctx.fill_(ctx0)
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record()
        ds.kv_append(x_new, n_new, kv, 1)
        b_.record()
        torch.cuda.synchronize()
        if k >= args.warmup:
            times.append(a_.elapsed_time(b_))
    assert ds.check() == 0 and int(ctx.item()) == ctx0 + n
    ms = statistics.median(times)
    nbytes = g.n_layers * (g.kv_dim * g.hidden * 2 + n * g.kv_dim * 2) + n * g.hidden * 4
    pk, src = peaks()
    print(json.dumps({"only": "append", "tokens": n, "layers": g.n_layers, "median_call_ms": ms,
                      "algorithmic_bytes": nbytes, "achieved_GBps": nbytes / (ms * 1e-3) / 1e9,
                      "peak_GBps": pk["hbm_gbs"], "peak_source": src}))


# ---------------------------------------------------------------------------
# Drift / acceptance-ceiling harness ("Kimi-K3-DSpark-NVFP4", Measurement and
# Detail): a weight format against the bf16 path on the same synthetic blocks.
# ---------------------------------------------------------------------------
def weight_snr_db(w_ref: torch.Tensor, w_dec: torch.Tensor) -> float:
    """10 log10(sum w^2 / sum (w - w_decoded)^2)."""
    w = w_ref.to(torch.float64)
    e = w - w_dec.to(torch.float64)
    return float(10.0 * torch.log10((w * w).sum() / (e * e).sum()))


def kl_and_overlap(l_ref: torch.Tensor, l_var: torch.Tensor):
    """Per row: KL(softmax(l_ref) || softmax(l_var)) and the coupling 1 - TV = sum min(p, q)."""
    lp = torch.log_softmax(l_ref.to(torch.float64), dim=-1)
    lq = torch.log_softmax(l_var.to(torch.float64), dim=-1)
    p = lp.exp()
    kl = (p * (lp - lq)).sum(-1)
    overlap = torch.minimum(p, lq.exp()).sum(-1)
    return kl, overlap


def prefix_runs(agree: np.ndarray) -> np.ndarray:
    """Length of the leading run of agreeing positions of every block ([N, B] bool)."""
    agree = np.asarray(agree, dtype=bool)
    run = np.cumprod(agree, axis=1)
    return run.sum(axis=1)


def conditional_agreement(agree: np.ndarray) -> np.ndarray:
    """s_i = P(position i agrees | positions < i agree), the per-position sequential agreement."""
    agree = np.asarray(agree, dtype=bool)
    s = []
    alive = np.ones(agree.shape[0], dtype=bool)
    for i in range(agree.shape[1]):
        n = alive.sum()
        s.append(float((alive & agree[:, i]).sum() / n) if n else 0.0)
        alive &= agree[:, i]
    return np.array(s)


def ceiling_from_agreement(s: np.ndarray) -> float:
    """Drift-limited acceptance ceiling sum_k prod_{i<=k} s_i (the expected leading run)."""
    return float(np.cumprod(np.asarray(s, dtype=np.float64)).sum())


def pearson(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    a = a - a.mean()
    b = b - b.mean()
    return float((a * b).sum() / np.sqrt((a * a).sum() * (b * b).sum()))


_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def decode_weight(v, fmt: str) -> torch.Tensor:
    """Decoded float64 matrix of a quantised weight triple (for the weight SNR)."""
    d, sc, g = v
    if fmt == "fp8":
        return d.view(torch.float8_e4m3fn).to(torch.float64) * sc.to(torch.float64)[:, None]
    codes = torch.stack([d & 0xF, d >> 4], dim=-1).reshape(d.shape[0], -1).long()
    vals = torch.tensor(_E2M1, dtype=torch.float64, device=d.device)[codes]
    if fmt == "nvfp4":
        return vals * sc.view(torch.float8_e4m3fn).to(torch.float64).repeat_interleave(16, 1) * g
    return vals * torch.pow(2.0, sc.to(torch.float64) - 127.0).repeat_interleave(32, 1)


def drift_harness(args):
    """Weight-format drift on the same kernels: every format against the bf16 path on the
    same blocks ("Kimi-K3-DSpark-NVFP4", Measurement / Detail). Aux regimes: gauss (N(0,1)),
    heavy (Student-t df 3 at unit RMS), boot (the drafter's own residual stream after each of
    its 5 layers, from a gauss block, stands in for the 5 captured target states). Greedy
    agreement, 1-TV and KL are teacher-forced (every format's logits corrected with the bf16
    path's previous tokens); the sequential agreement and the ceiling use every format's own
    greedy rollout. One JSON line per regime."""
    from dataclasses import replace
    import mla_block_diffusion_gb300 as M
    from mla_block_diffusion_gb300 import build as libbuild
    from synthetic import generate as gen
    from synthetic import quantize as Q
    from synthetic.configs import FULL_STEP, FORMAT_FP8, FORMAT_MXFP4, FORMAT_NVFP4
    libbuild.build()
    w = FULL_STEP
    G = w.geom
    if args.drift_geom == "mid":
        G = replace(G, hidden=1024, n_aux=5, n_heads=16, q_lora=512, kv_lora=512, d_nope=64, d_rope=64, d_v=64,
                    inter=2048, vocab=8192, rank=32)
        w = replace(w, geom=G, ctx=(512,))
    W = gen.make_weights(w, "cuda")
    I = gen.make_inputs(w, "cuda")
    ctx = I["ctx_list"][0]
    fmts = [f for f in args.drift_formats.split(",") if f]
    code = {"fp8": FORMAT_FP8, "nvfp4": FORMAT_NVFP4, "mxfp4": FORMAT_MXFP4}
    qnames = ["w_fc"] + [f"l{l}.{k}" for l in range(G.n_layers) for k in ("w_q_b", "w_o", "w_gate", "w_up", "w_down")]
    Wq, snr = {}, {}
    for f in fmts:
        Wq[f] = Q.quantise_weights(W, f, G.n_layers)
        num = den = 0.0
        for n in qnames:
            ref = W[n].to(torch.float64)
            dec = decode_weight(Wq[f][n], f)
            num += float((ref * ref).sum())
            den += float(((ref - dec) ** 2).sum())
            del ref, dec
        snr[f] = 10.0 * math.log10(num / den)
    handles = {"bf16": M.DSpark(G, W, max_bs=1, max_ctx=ctx)}
    for f in fmts:
        handles[f] = M.DSpark(G, Wq[f], max_bs=1, max_ctx=ctx, weight_format=code[f])
    depth = {}
    for k in range(1, G.n_layers + 1):  # the boot regime's residual streams
        Gk = replace(G, n_layers=k)
        depth[k] = M.DSpark(Gk, {n: t for n, t in W.items() if not n.startswith("l") or int(n[1:n.index(".")]) < k},
                            max_bs=1, max_ctx=ctx)
    kvs = {n: h.make_kv(I["kv_pools"], I["page_table"], I["ctx_len"], ctx) for n, h in handles.items()}
    kvd = {k: h.make_kv(I["kv_pools"], I["page_table"], I["ctx_len"], ctx) for k, h in depth.items()}
    w1 = W["markov_w1"].float()
    w2 = W["markov_w2"].float()
    smp = M.Sample(M.GREEDY, M.GREEDY, 1.0, 1.0, 1, 0)
    B, H, V = G.block, G.hidden, G.vocab
    x = torch.empty(1, B, H, dtype=torch.float32, device="cuda")
    h_out = torch.empty_like(x)
    z = torch.empty(1, B, V, dtype=torch.float32, device="cuda")
    ell = torch.empty_like(z)
    tok = torch.empty(1, B, dtype=torch.int32, device="cuda")
    conf = torch.empty(1, B, dtype=torch.float32, device="cuda")
    regimes = ["boot", "heavy", "gauss"] if args.regime == "all" else [args.regime]
    n_or = args.drift_oracle_blocks
    OW = None
    if n_or > 0:
        from oracle import build as obuild
        obuild.build()
        OW = OracleWeights(W, G)
    for regime in regimes:
        acc = {f: {"greedy": [], "seq": [], "kl": [], "ov": [], "hrel": [], "conf": []} for f in fmts}
        acc_or = {f: {"greedy": [], "seq": [], "hrel": []} for f in ["bf16"] + fmts}
        conf_ref = []
        t0 = time.time()
        for blk in range(args.blocks):
            seed = 7000 + blk
            if regime == "heavy":
                aux = gen.student_t3_unit_rms((1, B, G.n_aux, H), seed, "drift_aux", "cuda")
            else:
                aux = gen.normal((1, B, G.n_aux, H), 1.0, seed, "drift_aux", "cuda")
            if regime == "boot":
                layers_out = []
                for k in range(1, G.n_layers + 1):
                    depth[k].fuse_ctx(aux, x, 1)
                    depth[k].draft_block(x, kvd[k], h_out, z, 1)
                    layers_out.append(x.clone())
                aux = torch.stack(layers_out[:G.n_aux], dim=2).to(torch.bfloat16)
            anchor = gen.uniform_tokens((1,), V, seed, "drift_anchor").cuda()
            out = {}
            for n, hd in handles.items():
                hd.fuse_ctx(aux, x, 1)
                hd.draft_block(x, kvs[n], h_out, z, 1)
                hd.markov_rollout(z, anchor, smp, tok, ell, 1)
                hd.confidence(h_out, conf, 1)
                out[n] = (h_out[0].clone(), z[0].clone(), tok[0].clone(), conf[0].clone())
            if blk < n_or:
                # the float64 oracle on the same block: the FP32-class reference of the cards'
                # table, against which bf16 itself is the noise floor
                h_o, z_o, t_o = oracle_drift_block(OW, G, aux, I, ctx, int(anchor.item()))
                prev_o = torch.as_tensor(np.concatenate([[int(anchor.item())], t_o[:-1]]), device="cuda").long()
                delta_o = (w1[prev_o] @ w2).double().cpu().numpy()
                g_o = np.argmax(z_o + delta_o, axis=1)
                for n in ["bf16"] + fmts:
                    h_n, z_n, t_n, _ = out[n]
                    acc_or[n]["greedy"].append(np.argmax(z_n.double().cpu().numpy() + delta_o, axis=1) == g_o)
                    acc_or[n]["seq"].append(t_n.cpu().numpy() == t_o)
                    hn = h_n.double().cpu().numpy()
                    acc_or[n]["hrel"].append(float(np.linalg.norm(hn - h_o) / np.linalg.norm(h_o)))
            h_r, z_r, t_r, c_r = out["bf16"]
            prev = torch.cat([anchor.long(), t_r[:-1].long()])
            delta = w1[prev] @ w2                      # the Markov correction after the bf16 path's tokens
            l_r = z_r + delta
            conf_ref.append(c_r.cpu().numpy())
            for f in fmts:
                h_v, z_v, t_v, c_v = out[f]
                l_v = z_v + delta
                a = acc[f]
                a["greedy"].append((l_v.argmax(-1) == l_r.argmax(-1)).cpu().numpy())
                a["seq"].append((t_v == t_r).cpu().numpy())
                kl, ov = kl_and_overlap(l_r, l_v)
                a["kl"].append(kl.cpu().numpy())
                a["ov"].append(ov.cpu().numpy())
                a["hrel"].append(float(torch.linalg.norm(h_v - h_r) / torch.linalg.norm(h_r)))
                a["conf"].append(c_v.cpu().numpy())
        assert all(h.check() == 0 for h in list(handles.values()) + list(depth.values()))
        cr = np.concatenate(conf_ref)
        res = {}
        for f in fmts:
            a = acc[f]
            seq = np.stack(a["seq"])
            s_i = conditional_agreement(seq)
            kl = np.concatenate(a["kl"])
            cv = np.concatenate(a["conf"])
            res[f] = {"weight_snr_db": round(snr[f], 2),
                      "greedy_agreement": float(np.concatenate(a["greedy"]).mean()),
                      "sequential_rollout": float(seq.mean()),
                      "per_position_sequential": [round(float(v), 4) for v in s_i],
                      "ceiling": ceiling_from_agreement(s_i),
                      "mean_leading_run": float(prefix_runs(seq).mean()),
                      "one_minus_tv": float(np.concatenate(a["ov"]).mean()),
                      "kl_mean": float(kl.mean()), "kl_p99": float(np.percentile(kl, 99)),
                      "hidden_rel_err": float(np.mean(a["hrel"])),
                      "confidence_r": pearson(cr, cv),
                      "flip_rate": float(np.mean((cr > 0.5) != (cv > 0.5)))}
        vs_oracle = None
        if n_or > 0:
            vs_oracle = {}
            for n in ["bf16"] + fmts:
                seq = np.stack(acc_or[n]["seq"])
                s_i = conditional_agreement(seq)
                vs_oracle[n] = {"greedy_agreement": float(np.concatenate(acc_or[n]["greedy"]).mean()),
                                "sequential_rollout": float(seq.mean()),
                                "per_position_sequential": [round(float(v), 4) for v in s_i],
                                "ceiling": ceiling_from_agreement(s_i),
                                "hidden_rel_err": float(np.mean(acc_or[n]["hrel"]))}
        print(json.dumps({"drift": regime, "blocks": args.blocks, "geometry": args.drift_geom, "ctx": ctx,
                          "vs_float64_oracle": vs_oracle, "oracle_blocks": n_or,
                          "reference": "bf16 weights on the same kernels", "seconds": round(time.time() - t0, 1),
                          "formats": res}))


def oracle_drift_block(OW, G, aux, I, ctx, anchor):
    """The float64 oracle on one drift block (sequence 0's cache): h_out [B, H], z [B, V]
    and its own greedy Markov rollout from the anchor."""
    from oracle import network as N
    from oracle import sampling as S
    f64 = lambda t: t.detach().to(torch.float64).cpu().numpy()
    table = I["page_table"][0]
    pages = table[: (ctx + G.page_size - 1) // G.page_size].long()
    x = N.fuse_ctx(OW.get("w_fc"), f64(aux[0]))
    pos = np.arange(G.block, dtype=np.float64) + ctx
    for l in range(G.n_layers):
        L = {k: OW.get(f"l{l}.{k}") for k in LAYER_KEYS}
        pool = f64(I["kv_pools"][l][pages])
        cache = N.gather_cache(pool, np.arange(pool.shape[0]), ctx)
        x = N.layer(x, L, G, cache[:, :G.kv_lora], cache[:, G.kv_lora:], pos)
    h = N.rmsnorm(x, OW.get("final_norm"), G.eps)
    z = np.empty((G.block, G.vocab), dtype=np.float64)
    for lo, wl in OW.lm_chunks():
        z[:, lo:lo + wl.shape[0]] = h @ wl.T
    toks, _ = S.markov_rollout(z.astype(np.float32), OW.W["markov_w1"].cpu(), OW.W["markov_w2"].cpu(), anchor)
    return h, z, toks


def only_verify(args, G, local):
    """dspark_verify alone at the full vocabulary, bs=1: greedy, token-by-token probabilistic
    and block verification of one 7-token block (sampled draft, T 1, top_p 0.95). Target
    logits: the draft logits plus N(0, 0.5^2)."""
    from dataclasses import replace
    import mla_block_diffusion_gb300 as M
    from mla_block_diffusion_gb300 import build as libbuild
    from synthetic import generate as gen
    from synthetic.configs import FULL_STEP
    libbuild.build()
    torch.cuda.set_device(local)
    g = replace(G, hidden=64, n_aux=1, n_layers=1, n_heads=1, q_lora=64, kv_lora=64, d_nope=16, d_rope=16, d_v=64,
                inter=64)
    w = replace(FULL_STEP, geom=g)
    W = gen.make_weights(w, "cuda")
    ds = M.DSpark(g, W, max_bs=1)
    ell = gen.draft_logits(1, g.block, g.vocab, 5, device="cuda")
    P = torch.cat([ell, ell[:, -1:]], dim=1) + gen.noise((1, g.block + 1, g.vocab), 0.5, 5, "tn", device="cuda")
    tokens = torch.stack([torch.argmax(ell[0, i]) for i in range(g.block)]).to(torch.int32)[None].contiguous()
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    out = torch.empty(1, g.block + 1, dtype=torch.int32, device="cuda")
    res = {}
    for name, mode, dmode in (("greedy", M.GREEDY, M.GREEDY), ("token", M.PROBABILISTIC, M.PROBABILISTIC),
                              ("block", M.BLOCK, M.PROBABILISTIC)):
        times = []
        for k in range(args.warmup + args.steps):
            smp = M.Sample(dmode, mode, 1.0, 0.95, 11, k)
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record()
            ds.verify(P, ell, tokens, smp, acc, out, 1)
            b_.record()
            torch.cuda.synchronize()
            if k >= args.warmup:
                times.append(a_.elapsed_time(b_))
        # back to back (launches queued ahead, as in the step's graph): per-call device time
        n = max(args.steps, 10)
        smp = M.Sample(dmode, mode, 1.0, 0.95, 11, 0)
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a_.record()
        for _ in range(n):
            ds.verify(P, ell, tokens, smp, acc, out, 1)
        b_.record()
        torch.cuda.synchronize()
        assert ds.check() == 0
        res[name] = {"median_call_ms": statistics.median(times), "back_to_back_call_ms": a_.elapsed_time(b_) / n,
                     "accept_len_last": int(acc.item())}
    print(json.dumps({"only": "verify", "vocab": g.vocab, "block": g.block, "modes": res}))


def verify_launches(verify_mode: int) -> int:
    """Kernels of one dspark_verify call: greedy takes the row argmax and a finalize
    kernel; probabilistic the nucleus kernel and the accept-and-draw kernel; block
    verification the nucleus, residual-mass and decision kernels."""
    return {0: 2, 1: 2, 2: 3}[verify_mode]


def ds_launches_per_step(ds, bs: int = 1, draft_mode: int = 0, verify_mode: int = 0) -> int:
    """Kernels one draft-and-verify step launches (mirrors the library's choices).

    fc; per layer RMSNorm, q_a||kv_a, latent norms, q_b, q absorption, attention,
    split combine + v absorption (one fused kernel on the tensor-core path; two
    kernels otherwise when the KV sequence is split), o_proj, RMSNorm, gate/up,
    down; then the final RMSNorm, lm_head, rollout (one kernel), confidence and
    the verify kernels.
    """
    G = ds.G
    R = G.block * G.n_heads
    if G.kv_lora + G.d_rope == 576 and G.kv_lora == 512:  # tensor-core attention
        sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        tiles, parts = -(-R // 128), G.kv_lora // 256
        chunks = -(-ds.max_ctx // 64) + 1
        s = max(1, min(sms // (tiles * parts * ds.max_bs), chunks, 20))
        cps = -(-chunks // s)
        splits = -(-chunks // cps)
        fused = G.kv_lora % 64 == 0 and splits <= 20
        per_layer = 11 + (1 if splits > 1 and not fused else 0)
    else:
        per_layer = 11 + (1 if ds_layout_splits(ds) > 1 else 0)
    return 1 + G.n_layers * per_layer + 2 + 1 + 1 + verify_launches(verify_mode)


def ds_layout_splits(ds) -> int:
    """KV split count the library uses for this workload (mirrors its split rule)."""
    G = ds.G
    R = G.block * G.n_heads
    qtiles = (R + 63) // 64
    chunks = (ds.max_ctx + G.block + 63) // 64
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    want = -(-sms // (qtiles * ds.max_bs))
    cap = (chunks + 3) // 4
    s = max(1, min(want, cap, 64))
    cps = -(-chunks // s)
    return -(-chunks // cps)


if __name__ == "__main__":
    main()
