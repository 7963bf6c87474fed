#!/usr/bin/env python
"""Throughput of one Muon / Sign-Muon optimizer step on GB300, as one JSON line.

A step is the whole hot path over one batch of synthetic input resident in HBM:
  Muon:       momentum -> Newton–Schulz (bf16 tensor cores) -> W <- W - lr*U
  Sign-Muon:  momentum (per worker) -> Newton–Schulz with fused sign packing
              -> majority vote -> W <- W - lr*S_bar
              (--variant int8: int8 signs, integer sum, threshold; --post-polar:
              Newton–Schulz on S_bar before the update)
  Dion:       (--config 6) B = M + G, warm-started power iteration, error feedback,
              column normalisation, low-rank update
every stage through the C ABI of libmao.so.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl reference]
  python bench.py --sweep-hbm      (each HBM-bound kernel alone on L2-cold buffers)

Default workload: the 12-layer d=768 transformer-shaped Muon step (48 bf16 matrices). On
one GPU the default run also measures the other five workloads (64x128 Sign-Muon, 4096^2
Sign-Muon with 8 workers, the 32-layer dense model, the 128-expert MoE, the Dion step on the
12-layer shapes) and reports them under "per_config" (--no-per-config skips them).

Across N GPUs (torchrun) a Muon workload runs layer-wise: every matrix is owned by one rank
(longest-first on Newton–Schulz flops) and the updated weights are all-gathered; a Sign-Muon
workload splits its workers over the ranks and all-gathers the packed signs (or all-reduces
the int8 signs). The job's total work is fixed ("scaling": "strong"). Dion runs as replicas.

`--impl reference` times the fp64 CPU oracle on the same workload and metric on rank 0
only: whole steps where one takes seconds (the 64x128 and 12-layer workloads), otherwise
each step a bounded sample of the workload (its first matrices or workers), reported as
such.
"""

import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_STEPS = {1: 2000, 2: 400, 3: 60, 4: 10, 5: 100, 6: 400}
DEFAULT_WARMUP = {1: 20, 2: 10, 3: 5, 4: 3, 5: 5, 6: 10}
# workloads measured beside the default one (steps, warm-up steps), on one GPU
PER_CONFIG = {1: (2000, 20), 3: (60, 5), 4: (10, 3), 5: (100, 5), 6: (300, 10)}
PARITY_TESTS = {
    1: "tests/test_gpu_steps.py::test_config1_sign_muon_64x128_f32",
    2: "tests/test_gpu_steps.py::test_config2_muon_gpt12_d768_full, "
       "test_config2_fused_step_equals_composed_full",
    3: "tests/test_gpu_steps.py::test_config3_sign_muon_4096_w8_full",
    4: "tests/test_gpu_steps.py::test_config4_dense32_full",
    5: "tests/test_gpu_steps.py::test_config5_moe_grouped_full, "
       "test_config5_fused_step_equals_composed_full",
    6: "tests/test_gpu_steps.py::test_config6_dion_full",
}
# the oracle arm times whole steps when one step is at most this many dense NS flops
REFERENCE_WHOLE_STEP_FLOPS = 4e12
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# kernels timed over a window at least this long run under the power cap: sustained peak
SUSTAINED_WINDOW_S = 1.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5, 6])
    ap.add_argument("--impl", default="mao", choices=["mao", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work budget of the oracle baseline sample")
    ap.add_argument("--variant", default="bits", choices=["bits", "int8"],
                    help="Sign-Muon aggregation: 1-bit all-gather (bits) or int8 SUM all-reduce")
    ap.add_argument("--post-polar", action="store_true",
                    help="Sign-Muon: Newton-Schulz on the aggregated signs before the update")
    ap.add_argument("--sweep-hbm", action="store_true",
                    help="time each HBM-bound kernel alone on L2-cold buffers of 256 MB-4 GB "
                         "and print one JSON line per kernel and size")
    ap.add_argument("--block", default=None, metavar="ROWSxCOLS",
                    help="Muon workloads: blockwise Newton-Schulz, every ROWS x COLS block of "
                         "each matrix orthogonalised on its own")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of one captured CUDA graph of the step (the library's "
                         "calls are capture-safe)")
    ap.add_argument("--unfused", action="store_true",
                    help="Muon workloads: momentum, Newton-Schulz and update as three calls "
                         "instead of one muon_step call")
    ap.add_argument("--compute", default=None, choices=["bf16", "f32"],
                    help="Newton-Schulz arithmetic (default: the workload's): f32 is the "
                         "accuracy path (fp32 storage, FFMA products)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="do not measure the other workloads beside the default one")
    return ap.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def choose_peak(peaks, src, window_s):
    """The bf16 denominator of a tensor-core kernel timed over `window_s` seconds: the burst
    figure for a kernel timed alone in a short window, the sustained one for a window long
    enough to run under the power cap. Returns (peak, source text)."""
    if window_s >= SUSTAINED_WINDOW_S:
        return (peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]),
                "%s bf16_tflops_sustained (per-launch timing window %.2f s >= %.0f s)"
                % (src, window_s, SUSTAINED_WINDOW_S))
    return (peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]),
            "%s bf16_tflops burst (per-launch timing window %.2f s < %.0f s)"
            % (src, window_s, SUSTAINED_WINDOW_S))


def fp32_peak_tflops(dev):
    """fp32 FFMA peak of the device: SMs x 128 lanes x 2 flops x the maximum SM clock."""
    import torch
    props = torch.cuda.get_device_properties(dev)
    peaks, _ = load_peaks()
    mhz = peaks.get("sm_max_mhz", 2070.0)
    return props.multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12


# ------------------------------------------------------------------ work model

def alg_flops(shapes, steps):
    """Newton–Schulz flops the method needs given symmetric A and B:
    m(m+1)n (A = X X^T) + m^2(m+1) (A A) + 2 m^2 n (B X) per iteration."""
    tot = 0
    for R, C in shapes:
        m, n = min(R, C), max(R, C)
        tot += steps * (m * (m + 1) * n + m * m * (m + 1) + 2 * m * m * n)
    return tot


def dense_flops(shapes, steps):
    """(4 m^2 n + 2 m^3) per iteration (dense count)."""
    tot = 0
    for R, C in shapes:
        m, n = min(R, C), max(R, C)
        tot += steps * (4 * m * m * n + 2 * m ** 3)
    return tot


def esize(dt):
    import torch
    return 2 if dt == torch.bfloat16 else 4


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ the step

class Step:
    """Device buffers and the sequence of C-ABI calls of one optimizer step."""

    def __init__(self, wl, inputs, device, variant="bits", post_polar=False, block=None,
                 fused=True, dplan=None):
        """variant: "bits" (1-bit all-gather) or "int8" (integer SUM all-reduce) aggregation
        of a Sign-Muon workload; post_polar: the optional Newton–Schulz step on S_bar;
        fused: a Muon workload on the tensor cores runs as one muon_step call (momentum in
        the staging pass, the update in the last product) instead of the three calls;
        dplan: the step across ranks (distributed.LayerwiseMuon for a Muon workload,
        distributed.SignExchange for a Sign-Muon workload), None on one GPU."""
        import torch
        import matrix_aware_optimizers_gb300 as mao
        if wl.kind != "sign" and (variant != "bits" or post_polar):
            raise ValueError("the aggregation variants apply to Sign-Muon workloads only")
        if variant not in ("bits", "int8"):
            raise ValueError(variant)
        if block is not None and wl.kind != "muon":
            raise ValueError("blockwise Newton-Schulz applies to the Muon workloads")
        self.mao = mao
        self.wl = wl
        self.variant, self.post_polar = variant, post_polar
        self.block = block
        self.fused = fused and wl.kind == "muon" and block is None and wl.compute == "bf16"
        # Sign-Muon, 1-bit variant: the four stages as one sign_muon_step call
        self._sign_call = {}  # prepared sign_muon_step calls by stream
        self._current_stream = torch.cuda.current_stream
        self.fused_sign = fused and wl.kind == "sign" and variant == "bits" and not post_polar \
            and dplan is None
        self.W, self.M, self.G = inputs["W"], inputs["M"], inputs["G"]
        self.dev = device
        self.dplan = dplan
        if dplan is not None:
            self._init_dist(wl, device, variant, post_polar, block)
            return
        if wl.kind == "dion":
            # one Dion step per call: the previous right factors Q are updated in place
            self.Q = inputs["Q"]
            self.U = []
            need = mao.dion_workspace_bytes([tuple(w.shape) for w in self.W], wl.rank)
            self.ws = torch.empty(need, dtype=torch.uint8, device=device)
            return
        if wl.kind == "sign":
            R, C = self.W[0].shape
            self.nbits = R * C
            nw = mao.packed_words(R, C)
            stride = (nw + 3) // 4 * 4
            self.vote = torch.zeros(stride, dtype=torch.int32, device=device)
            if variant == "bits":
                self.words = torch.zeros((wl.workers, stride), dtype=torch.int32, device=device)
                self.bits = [self.words[m, :nw] for m in range(wl.workers)]
                self.U = [None] * wl.workers
            else:
                # U of each worker, then its int8 signs in the all-reduce buffer layout
                self.U = [torch.empty_like(m) for m in self.M]
                s_stride = (self.nbits + 15) // 16 * 16
                self.s8 = torch.zeros((wl.workers, s_stride), dtype=torch.int8, device=device)
                self.sbar = torch.zeros(self.nbits, dtype=torch.int8, device=device)
            if post_polar:
                self.U_bar = torch.empty_like(self.W[0])
        elif not self.fused:
            self.U = [torch.empty_like(w) for w in self.W]
        else:
            self.U = []
        if block is not None:
            n = mao.ns_blockwise_workspace_bytes(self.M, block, wl.compute)
            self.ws = torch.empty(n, dtype=torch.uint8, device=device)
        else:
            self.ws = mao.workspace(self.M, wl.compute, device)

    def momentum(self):
        if self.wl.kind == "dion":  # B = M + G is the first stage of the Dion call
            return
        self.mao.muon_momentum_update(self.M, self.G, self.wl.mu)

    def ns(self):
        wl = self.wl
        if wl.kind == "dion":
            self.mao.dion_step(self.W, self.M, self.G, self.Q, wl.mu, wl.lr, ws=self.ws)
            return
        if self.block is not None:
            self.mao.ns_orthogonalize_blockwise(self.M, self.U, self.block, wl.steps, wl.coeffs,
                                                wl.eps, wl.compute, ws=self.ws)
            return
        if wl.kind == "sign" and self.variant == "bits":
            self.mao.ns_orthogonalize(self.M, self.U, wl.steps, wl.coeffs, wl.eps, wl.compute,
                                      sign_bits=self.bits, ws=self.ws)
        else:
            self.mao.ns_orthogonalize(self.M, self.U, wl.steps, wl.coeffs, wl.eps, wl.compute,
                                      ws=self.ws)
            if wl.kind == "sign":
                for m in range(wl.workers):
                    self.mao.sign_int8(self.U[m], self.s8[m, : self.nbits].view(self.U[m].shape))

    def update(self):
        wl = self.wl
        if wl.kind == "dion":  # the updates of M and X are the last stages of the Dion call
            return
        if wl.kind != "sign":
            self.mao.apply_update(self.W, wl.lr, U=self.U)
            return
        if self.variant == "bits":
            self.mao.majority_vote_packed(self.words, self.nbits, self.vote)
            s_bar = self.mao.PackedSigns(self.vote, *self.W[0].shape)
        else:
            self.mao.majority_vote_int8(self.s8, self.nbits, s_bar=self.sbar if self.post_polar else None,
                                        vote=None if self.post_polar else self.vote)
            s_bar = self.sbar.view(self.W[0].shape)
        if self.post_polar:
            self.mao.ns_orthogonalize(s_bar, self.U_bar, wl.steps, wl.coeffs, wl.eps, wl.compute,
                                      ws=self.ws)
            self.mao.apply_update(self.W, wl.lr, U=self.U_bar)
        else:
            self.mao.apply_update(self.W, wl.lr, vote=self.vote)

    def fused_call(self, W_out=None):
        """The one-call step (muon_step, or dion_step for Dion) writing the new weights to
        W_out (None: in place)."""
        wl = self.wl
        if wl.kind == "dion":
            self.mao.dion_step(self.W, self.M, self.G, self.Q, wl.mu, wl.lr, ws=self.ws,
                               X_out=W_out)
            return
        self.mao.muon_step(self.W, self.M, self.G, wl.mu, wl.lr, wl.steps, wl.coeffs, wl.eps,
                           wl.compute, ws=self.ws, W_out=W_out)

    def _init_dist(self, wl, device, variant, post_polar, block):
        import torch
        from matrix_aware_optimizers_gb300 import distributed
        mao, plan = self.mao, self.dplan
        if block is not None or post_polar:
            raise ValueError("the step across ranks runs without blocks or the post-vote polar step")
        if wl.kind == "muon":
            if not self.fused:
                raise ValueError("the layer-wise step runs the one-call muon_step")
            # every rank holds every weight (the layout of the all-gather); momenta and
            # gradients only of the matrices it owns
            self.flat, views = plan.layout.allocate(device)
            for v, w in zip(views, self.W):
                v.copy_(w)
            self.W = views
            self.M = [self.M[i] for i in plan.mine]
            self.G = [self.G[i] for i in plan.mine]
            self.U = []
            self.ws = mao.workspace(self.M, wl.compute, device) if self.M else None
            self.shapes_own = [tuple(m.shape) for m in self.M]
            return
        if wl.kind != "sign":
            raise ValueError("Dion runs as replicas across ranks")
        ex = plan
        mine = range(ex.first_worker, ex.first_worker + ex.local)
        self.M = [self.M[m] for m in mine]
        self.G = [self.G[m] for m in mine]
        self.nbits = ex.nbits
        self.vote = torch.zeros(ex.stride, dtype=torch.int32, device=device)
        if variant == "bits":
            self.words = ex.allocate_words(device)
            self.bits = ex.my_words(self.words)
            self.U = [None] * ex.local
        else:
            self.U = [torch.empty_like(m) for m in self.M]
            self.s8 = torch.zeros((ex.local, ex.s_stride), dtype=torch.int8, device=device)
            self.total = torch.zeros(ex.nbits, dtype=torch.int8, device=device)
        self.ws = mao.workspace(self.M, wl.compute, device)
        self.shapes_own = [tuple(m.shape) for m in self.M]
        self._distributed = distributed

    def dist_call(self):
        """One step of this rank across ranks: its share of the work, then the exchange."""
        from matrix_aware_optimizers_gb300 import distributed
        wl, plan = self.wl, self.dplan
        if wl.kind == "muon":
            if self.M:
                self.mao.muon_step([self.W[i] for i in plan.mine], self.M, self.G, wl.mu, wl.lr,
                                   wl.steps, wl.coeffs, wl.eps, wl.compute, ws=self.ws)
            distributed.allgather_weights(plan.layout, self.flat, plan.group)
        elif self.variant == "bits":
            distributed.sign_muon_step(plan, self.W[0], self.M, self.G, self.words, self.vote,
                                       wl.mu, wl.lr, wl.steps, wl.coeffs, wl.eps, wl.compute,
                                       ws=self.ws)
        else:
            distributed.sign_muon_step_int8(plan, self.W[0], self.M, self.G, self.U, self.s8,
                                            self.total, self.vote, wl.mu, wl.lr, wl.steps,
                                            wl.coeffs, wl.eps, wl.compute, ws=self.ws)

    @property
    def whole_call(self):
        """The step is one call (or one call and its exchange): no per-stage timing."""
        return self.fused or self.fused_sign or self.dplan is not None

    def __call__(self):
        if self.dplan is not None:
            self.dist_call()
            return
        if self.fused:
            self.fused_call()
            return
        if self.fused_sign:
            # the call's arguments marshalled once per stream (the tensors keep their
            # storage), as a training loop would hold them
            key = self._current_stream().cuda_stream
            call = self._sign_call.get(key)
            if call is None:
                wl = self.wl
                call = self.mao.sign_muon_step(
                    self.W[0], self.M, self.G, self.words, self.vote, wl.mu, wl.lr, wl.steps,
                    wl.coeffs, wl.eps, wl.compute, ws=self.ws, prepare=True)
                self._sign_call[key] = call
            call()
            return
        self.momentum()
        self.ns()
        self.update()


def stage_bytes(wl, step):
    """Algorithmic HBM bytes of the elementwise stages per step (the update stage's figure is
    None when it holds the post-vote Newton–Schulz, which is not elementwise)."""
    mom = sum(m.numel() * (2 * esize(m.dtype) + esize(g.dtype)) for m, g in zip(step.M, step.G))
    if wl.kind == "sign" and step.post_polar:
        upd = None
    elif wl.kind == "sign" and step.variant == "int8":
        n = step.nbits  # W_n int8 signs read, packed vote written and read, W read + written
        upd = sum(w.numel() * 2 * esize(w.dtype) for w in step.W) + 2 * (n // 8) + wl.workers * n
    elif wl.kind == "sign":
        n = step.nbits
        upd = sum(w.numel() * 2 * esize(w.dtype) for w in step.W) + n // 8 + wl.workers * n // 8
    else:
        upd = sum(w.numel() * (2 * esize(w.dtype) + esize(u.dtype)) for w, u in zip(step.W, step.U))
    return mom, upd


# ------------------------------------------------------------------ oracle arm

def oracle_sample(wl, host, budget_s, max_items=None, variant="bits", post_polar=False,
                  block=None):
    """Time the fp64 oracle on whole matrices of the workload (cycling) for ~budget_s.

    Returns (fraction of one step processed, seconds, description)."""
    import numpy as np

    import oracle
    shapes = [tuple(x.shape) for x in host["M"]] if wl.kind != "sign" else [tuple(host["W"][0].shape)]
    # the fraction is of the workload's whole step (host may hold only a prefix of it)
    total = dense_flops(wl.shapes, wl.steps) * (wl.workers + (1 if post_polar else 0)
                                                if wl.kind == "sign" else 1)
    if wl.kind == "dion":  # work fraction by matrix elements (every element costs 8 r flops)
        total = sum(r * c for r, c in wl.shapes)
    store = "bf16" if wl.m_dtype.itemsize == 2 else "f32"
    wstore = "bf16" if wl.w_dtype.itemsize == 2 else "f32"
    done_flops, t_used, items = 0, 0.0, 0
    n_items = len(host["M"])
    words = {}
    i = 0
    while True:
        t0 = time.perf_counter()
        if wl.kind == "dion":
            oracle.dion_step(host["W"][i], host["M"][i], host["G"][i], host["Q"][i], wl.mu, wl.lr)
            done_flops += shapes[i][0] * shapes[i][1]
        elif wl.kind == "muon" and block is not None:
            M = oracle.momentum(host["M"][i], host["G"][i], wl.mu, store)
            U = oracle.blockwise_newton_schulz(M, block[0], block[1], wl.steps, wl.coeffs, wl.eps)
            oracle.apply_update_f64(host["W"][i], U, wl.lr)
            done_flops += dense_flops([shapes[i]], wl.steps)
        elif wl.kind == "muon":
            oracle.muon_step([host["W"][i]], [host["M"][i]], [host["G"][i]], wl.mu, wl.lr,
                             wl.steps, wl.coeffs, wl.eps, m_store=store)
            done_flops += dense_flops([shapes[i]], wl.steps)
        else:
            # one worker's momentum + NS + sign/pack; the vote and update run with the last
            M = oracle.momentum(host["M"][i], host["G"][i], wl.mu, store)
            U = oracle.newton_schulz(M, wl.steps, wl.coeffs, wl.eps)
            S_m = oracle.sign_of(U)
            words[i] = oracle.pack_signs(S_m) if variant == "bits" else S_m
            done_flops += dense_flops(shapes, wl.steps)
            if i == n_items - 1 and len(words) == n_items:
                if variant == "bits":
                    vote = oracle.majority_vote(np.stack([words[m] for m in range(n_items)]), U.size)
                    S = oracle.unpack_signs(vote, U.size).reshape(U.shape)
                else:
                    S = oracle.int8_sum_vote([words[m] for m in range(n_items)])[1]
                if post_polar:
                    U_bar = oracle.post_vote_polar(S, wl.steps, wl.coeffs, wl.eps)
                    oracle.apply_update_f64(host["W"][0], U_bar, wl.lr)
                else:
                    oracle.apply_update(host["W"][0], S, wl.lr, wstore)
        t_used += time.perf_counter() - t0
        items += 1
        i = (i + 1) % n_items
        if t_used >= budget_s or (max_items is not None and items >= max_items):
            break
    frac = done_flops / total
    desc = "%d matrix step(s) of the workload (%.3f of one step), fp64 numpy" % (items, frac)
    if wl.kind == "dion":
        desc += " (fraction by matrix elements)"
    return frac, t_used, desc


def blas_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        n = [d.get("num_threads") for d in info if d.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count()


def host_copy(inputs):
    return {k: [t.float().cpu().numpy() for t in v] for k, v in inputs.items()}


def reference_items(wl, post_polar=False):
    """Matrices (Muon, Dion) or workers (Sign-Muon) one timed oracle step covers: all of
    them when the whole step costs at most REFERENCE_WHOLE_STEP_FLOPS dense Newton–Schulz
    flops, else the longest prefix within that (at least one)."""
    if wl.kind == "dion":
        return len(wl.shapes)
    if wl.kind == "sign":
        per = dense_flops(wl.shapes, wl.steps)
        n_all = wl.workers
        if per * (n_all + (1 if post_polar else 0)) <= REFERENCE_WHOLE_STEP_FLOPS:
            return n_all
        return max(1, int(REFERENCE_WHOLE_STEP_FLOPS // per))
    tot, n = 0, 0
    for s in wl.shapes:
        tot += dense_flops([s], wl.steps)
        if n >= 1 and tot > REFERENCE_WHOLE_STEP_FLOPS:
            break
        n += 1
    return n


def run_reference(args, wl, block=None):
    """The oracle arm: the fp64 CPU oracle timed on the host cores, on rank 0 only, for the
    same workload, metric and config as the GPU arm."""
    from matrix_aware_optimizers_gb300 import workloads
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
    if rank != 0:
        return
    K = args.steps if args.steps is not None else 3
    Wu = args.warmup if args.warmup is not None else 1
    shapes = None
    if wl.index == 4:  # the oracle needs host copies of the inputs: generate one layer
        shapes = [(4096, 4096)] * 4 + [(4096, 14336), (14336, 4096), (4096, 14336)]
    inputs = workloads.generate(wl, "cpu", shapes=shapes)
    host = host_copy(inputs)
    var = dict(variant=args.variant, post_polar=args.post_polar, block=block)
    items = reference_items(wl, args.post_polar)
    whole = items == (wl.workers if wl.kind == "sign" else len(wl.shapes))
    for _ in range(Wu):  # warm-up: one matrix (or worker) each
        oracle_sample(wl, host, float("inf"), max_items=1, **var)
    frac, secs = 0.0, 0.0
    t0 = time.perf_counter()
    for _ in range(K):
        f, s, _ = oracle_sample(wl, host, float("inf"), max_items=items, **var)
        frac += f
        secs += s
    wall = time.perf_counter() - t0
    value = frac / secs
    if whole:
        sample = ("whole steps: every matrix (or worker) of the workload per timed step, fp64 "
                  "numpy momentum + Newton-Schulz + update (+ sign, vote)")
    else:
        sample = ("each timed step: the first %d %s of the workload (%.4f of one step), fp64 "
                  "numpy; value = work done / time, ms_per_step = time per timed step"
                  % (items, "workers" if wl.kind == "sign" else "matrices", frac / K))
    line = {
        "impl": "reference", "metric": metric_name(wl), "value": value, "unit": "steps/s",
        "n_gpus": args.gpus, "steps": K, "warmup": Wu, "ms_per_step": 1000.0 * wall / K,
        "higher_is_better": True, "scaling": scaling_of(wl, world), "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": config_block(wl, args.variant, args.post_polar, block, world),
        "step_fraction": frac / K,
        "warmup_sample": "one matrix (or worker) per warm-up step",
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": blas_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def reduce_max(x, device, world):
    """Max of a scalar over all ranks (identity at world size 1)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def scaling_of(wl, world):
    """Across ranks a Muon or Sign-Muon step splits one fixed step (strong scaling); Dion
    runs one copy per rank (weak). One GPU: strong (nothing is split)."""
    return "weak" if (wl.kind == "dion" and world > 1) else "strong"


def job_throughput(ms_max, steps, world, scaling="weak"):
    """Whole-job steps/s over the slowest rank's time: with weak scaling every rank steps
    its own copy of the workload (world * steps steps), with strong scaling the ranks
    together take `steps` steps."""
    n = world * steps if scaling == "weak" else steps
    return n / (ms_max / 1000.0)


def metric_name(wl):
    if wl.kind == "dion":
        return "Dion steps/s (%s)" % wl.name
    return ("Sign-Muon steps/s" if wl.kind == "sign" else "Muon steps/s") + \
        " (%s); NS TFLOP/s; elementwise GB/s" % wl.name


def dion_min_bytes(step):
    """Bytes a Dion step must move: read X, M, G and Q_prev; write X, M and Q."""
    tot = 0
    for x, m, g, q in zip(step.W, step.M, step.G, step.Q):
        tot += x.numel() * 2 * esize(x.dtype) + m.numel() * 2 * esize(m.dtype)
        tot += g.numel() * esize(g.dtype) + 2 * q.numel() * 4
    return tot


def touched_bytes(wl):
    """Bytes of the step's matrices read and written once (M of every worker, and W)."""
    n_m = wl.elements * (wl.workers if wl.kind == "sign" else 1)
    return 2 * n_m * esize(wl.m_dtype) + 2 * wl.elements * esize(wl.w_dtype)


def parallelism_of(wl, world):
    if world == 1:
        return "one GPU"
    if wl.kind == "muon":
        return ("layer-wise over %d ranks: whole matrices per rank (longest first on "
                "Newton-Schulz flops), then an all-gather(v) of the updated weights" % world)
    if wl.kind == "sign":
        return ("%d workers split over %d ranks; packed signs all-gathered (int8 variant: "
                "SUM all-reduce), vote and update on every rank" % (wl.workers, world))
    return "replicas: each of %d ranks steps its own copy of the workload" % world


def config_block(wl, variant="bits", post_polar=False, block=None, world=1):
    """The workload's description, identical for the GPU arm and the oracle arm."""
    c = {"workload": wl.name, "kind": wl.kind, "matrices": len(wl.shapes),
         "elements": wl.elements, "workers": wl.workers, "ns_steps": wl.steps,
         "coeffs": list(wl.coeffs), "mu": wl.mu, "lr": wl.lr, "compute": wl.compute,
         "parallelism": parallelism_of(wl, world)}
    tb = touched_bytes(wl)
    if tb > L2_BYTES:
        c["l2"] = "inputs larger than L2: %.0f MB of matrices touched per step vs 129 MB L2" % (tb / 1e6)
    else:
        c["l2"] = ("inputs smaller than L2 (%.2f MB touched per step, not flushed): the step "
                   "is launch-latency bound" % (tb / 1e6))
    if wl.kind == "sign":
        c["aggregation"] = ("1-bit packed all-gather + local vote" if variant == "bits" else
                            "int8 SUM all-reduce + local threshold")
        c["post_vote_polar"] = bool(post_polar)
    if wl.kind == "dion":
        c["rank"] = wl.rank
    if block is not None:
        c["blockwise"] = "%dx%d blocks" % tuple(block)
    return c


# ------------------------------------------------------------------ HBM sweep

def sweep_hbm(dev, reps=20):
    """GB/s of each HBM-bound kernel alone, on buffers far larger than L2 or rotated across
    >= 4 x L2 of distinct memory, so that every timed call reads cold lines."""
    import torch
    import matrix_aware_optimizers_gb300 as mao
    stream = torch.cuda.current_stream()
    peaks, src = load_peaks()
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    Wn = 8
    kernels = {
        # name: (bytes per element, setup(n) -> callable)
        "momentum bf16 M, bf16 G": 6,
        "momentum fp32 M, bf16 G": 10,
        "update Muon bf16 W, bf16 U": 6,
        "update Sign-Muon bf16 W, packed vote": 4 + 1 / 8,
        "sign_pack_bits bf16 U": 2 + 1 / 8,
        "sign_int8 bf16 U": 3,
        "majority_vote_packed 8 workers": (Wn + 1) / 8,
        "majority_vote_int8 8 workers": Wn + 1 / 8,
    }

    def make(name, n):
        C = 4096
        R = max(1, n // C)
        bf, f32 = torch.bfloat16, torch.float32
        if name.startswith("momentum"):
            M = torch.zeros((R, C), dtype=f32 if "fp32" in name else bf, device=dev)
            G = torch.ones((R, C), dtype=bf, device=dev)
            return lambda: mao.muon_momentum_update(M, G, 0.95)
        if name.startswith("update Muon"):
            W = torch.zeros((R, C), dtype=bf, device=dev)
            U = torch.ones((R, C), dtype=bf, device=dev)
            return lambda: mao.apply_update(W, 0.02, U=U)
        if name.startswith("update Sign"):
            W = torch.zeros((R, C), dtype=bf, device=dev)
            v = torch.zeros(mao.packed_words(R, C), dtype=torch.int32, device=dev)
            return lambda: mao.apply_update(W, 0.02, vote=v)
        if name.startswith("sign_pack"):
            U = torch.ones((R, C), dtype=bf, device=dev)
            b = torch.empty(mao.packed_words(R, C), dtype=torch.int32, device=dev)
            return lambda: mao.sign_pack_bits(U, b)
        if name.startswith("sign_int8"):
            U = torch.ones((R, C), dtype=bf, device=dev)
            s8 = torch.empty((R, C), dtype=torch.int8, device=dev)
            return lambda: mao.sign_int8(U, s8)
        if name.startswith("majority_vote_packed"):
            nw = mao.packed_words(R, C)
            words = torch.zeros((Wn, nw), dtype=torch.int32, device=dev)
            vote = torch.empty(nw, dtype=torch.int32, device=dev)
            return lambda: mao.majority_vote_packed(words, R * C, vote)
        s8 = torch.ones((Wn, R * C), dtype=torch.int8, device=dev)
        vote = torch.empty(mao.packed_words(R, C), dtype=torch.int32, device=dev)
        return lambda: mao.majority_vote_int8(s8, R * C, vote=vote)

    for name, bpe in kernels.items():
        for total in (256 << 20, 1 << 30, 4 << 30):
            n = int(total / bpe) // 4096 * 4096
            copies = max(1, -(-4 * L2_BYTES // total))  # rotate over >= 4 x L2 of memory
            fns = [make(name, n) for _ in range(copies)]
            for f in fns:
                f()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for r in range(reps):
                fns[r % copies]()
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / reps
            gbs = n * bpe / (ms / 1000.0) / 1e9
            print(json.dumps({"kernel": name, "bytes_per_call": int(n * bpe), "copies": copies,
                              "elements": n, "ms": ms, "GB/s": gbs, "peak_GB/s": hbm,
                              "frac": gbs / hbm, "peak_source": "%s hbm_gbs" % src}))
            del fns
            torch.cuda.empty_cache()


# ------------------------------------------------------------------ main arm

def _tc_launches_per_step(wl, step, block, post_polar):
    """Tensor-core (and Dion CUDA-core) launches of one step, for the profiling capacity."""
    if wl.kind == "dion":  # four products per round of shapes, set-up and CUDA-core kernels
        return 4 * ((len(set(wl.shapes)) + 7) // 8) + (len(wl.shapes) + 95) // 96 + 16
    shapes = getattr(step, "shapes_own", None) or [tuple(m.shape) for m in step.M]
    if block is not None:
        shapes = {(min(block[0], R - i), min(block[1], C - j)) for R, C in set(shapes)
                  for i in range(0, R, block[0]) for j in range(0, C, block[1])}
    return 3 * wl.steps * ((len(set(shapes)) + 7) // 8 + (1 if post_polar else 0))


def measure(opts, wl, dev, world, rank, local, block, K, Wu, barrier, max_over_ranks):
    """Time K steps of workload `wl` (after Wu warm-up steps) and the per-launch and
    per-stage passes after them; returns (bench line without e2e / CPU baseline, step)."""
    import torch
    import matrix_aware_optimizers_gb300 as mao
    from matrix_aware_optimizers_gb300 import distributed, workloads

    dplan = None
    seed = wl.index - 1
    if world > 1:
        if wl.kind == "muon" and block is None and not opts.unfused:
            dplan = distributed.LayerwiseMuon(wl.shapes, wl.w_dtype, wl.steps)
        elif wl.kind == "sign" and not opts.post_polar and wl.workers % world == 0:
            dplan = distributed.SignExchange(wl.shapes[0][0], wl.shapes[0][1], wl.workers)
        else:
            seed += 1000 * rank  # replicas: every rank its own copy
    scaling = "strong" if (world == 1 or dplan is not None) else "weak"
    inputs = workloads.generate(wl, dev, seed=seed)
    step = Step(wl, inputs, dev, opts.variant, opts.post_polar, block, fused=not opts.unfused,
                dplan=dplan)
    del inputs
    stream = torch.cuda.current_stream()

    for _ in range(Wu):
        step()
    mao.sync_status()
    run = step
    per_replay = None
    if opts.graph:  # one captured step, replayed (no host launch work per step)
        if dplan is not None:
            raise ValueError("--graph runs on one GPU")
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        captured0 = mao.launch_count()
        with torch.cuda.graph(graph, stream=side):
            step()
        torch.cuda.synchronize()
        per_replay = mao.launch_count() - captured0  # kernels of the library in one replay
        run = graph.replay
        for _ in range(Wu):
            run()
        mao.sync_status()

    # ---------------- timed region: K whole steps, inputs resident in HBM
    n_tc_per_step = _tc_launches_per_step(wl, step, block, opts.post_polar)
    launches0 = mao.launch_count()
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    launches = mao.launch_count() - launches0
    if per_replay is not None:  # replays launch the captured kernels without host calls
        launches = per_replay * K
    mao.sync_status()
    ms_total = max_over_ranks(e0.elapsed_time(e1))
    ms_step = ms_total / K
    value = job_throughput(ms_total, K, world, scaling)

    # ---------------- kernel-timing pass: the same steps with a CUDA event pair around every
    # tensor-core launch (on its stream). Kept out of the timed region above: an event
    # between two launches stops the next launch's set-up from overlapping the previous
    # kernel (programmatic dependent launch), and the records themselves cost time.
    reps_tc = max(3, min(K, 50))
    mao.profile_begin(reps_tc * n_tc_per_step)
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(reps_tc):
        step()
    p1.record(stream)
    torch.cuda.synchronize()
    tagged = mao.profile_end_tagged()
    mao.sync_status()
    ms_prof = p0.elapsed_time(p1)
    tc_ms = [ms for ms, tag in tagged if tag == "tc"]
    kernel_ms = {}  # per launch kind: milliseconds per step
    for ms, tag in tagged:
        kernel_ms[tag] = kernel_ms.get(tag, 0.0) + ms / reps_tc
    # the same steps with one event pair around each Newton–Schulz call's run of tensor-core
    # products instead: the products keep overlapping one another's set-up (programmatic
    # dependent launch), as in the timed region, so the run's span is the kernel's time
    # inside the step
    span_ms = None
    if wl.kind != "dion" and wl.compute == "bf16" and tc_ms:
        mao.profile_span_begin(reps_tc * 4)
        for _ in range(reps_tc):
            step()
        torch.cuda.synchronize()
        spans = mao.profile_span_end()
        mao.sync_status()
        if spans:
            span_ms = sum(spans) / reps_tc  # per step

    # ---------------- per-stage times (separate pass, same stream)
    reps = max(3, min(K, 50))
    if step.whole_call:
        # one call: the Newton–Schulz share is the tensor-core launches' time from the pass
        # above (the momentum rides on the staging pass, the update on the last product)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
        for r in range(reps):
            ev[r][0].record(stream)
            step()
            ev[r][1].record(stream)
        torch.cuda.synchronize()
        st_step = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
        st_mom = st_upd = None
        # the Newton–Schulz share: the tensor-core launches, or the one-launch fp32 kernel
        st_ns = sum(tc_ms) / reps_tc if tc_ms else kernel_ms.get("ns_small", st_step)
    else:
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps)]
        for r in range(reps):
            ev[r][0].record(stream)
            step.momentum()
            ev[r][1].record(stream)
            step.ns()
            ev[r][2].record(stream)
            step.update()
            ev[r][3].record(stream)
        torch.cuda.synchronize()
        st_mom = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
        st_ns = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
        st_upd = statistics.median(e[2].elapsed_time(e[3]) for e in ev)

    peaks, peak_src = load_peaks()
    cfg = config_block(wl, opts.variant, opts.post_polar, block, world)
    launch = {"launch": "CUDA graph replay" if opts.graph else "eager"}
    if wl.kind == "dion":
        line = dion_line(wl, step, K, Wu, world, value, ms_step, reps_tc, ms_prof, st_ns, tc_ms,
                         launches, clk, peaks, peak_src, cfg, scaling, kernel_ms=kernel_ms)
        line["step"] = launch
        return line, step

    # ---------------- roofline of the dominant kernel (tensor-core NS product kernel)
    shapes = getattr(step, "shapes_own", None) or [tuple(m.shape) for m in step.M]
    if block is not None:  # the products run on the blocks
        shapes = [(min(block[0], R - i), min(block[1], C - j)) for R, C in shapes
                  for i in range(0, R, block[0]) for j in range(0, C, block[1])]
    alg = alg_flops(shapes, wl.steps)
    dense = dense_flops(shapes, wl.steps)
    # the post-vote polar step is one more Newton–Schulz on a matrix of W's shape
    alg_tc = alg + (alg_flops([tuple(step.W[0].shape)], wl.steps) if opts.post_polar else 0)
    tc_total_ms = sum(tc_ms)
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    if wl.compute == "bf16" and tc_ms:
        per_step = len(tc_ms) / reps_tc
        iso_tflops = alg_tc * reps_tc / (tc_total_ms / 1000.0) / 1e12
        tflops = alg_tc / (span_ms / 1000.0) / 1e12 if span_ms else iso_tflops
        peak, peak_text = choose_peak(peaks, peak_src, ms_prof / 1000.0)
        roof = {"kernel": "ns_tc_kernel", "bound": "tensor", "achieved": tflops, "peak": peak,
                "unit": "TFLOP/s", "frac": tflops / peak, "traffic": None,
                "peak_source": peak_text,
                "work": "symmetric-minimum flops m(m+1)n + m^2(m+1) + 2m^2n per iteration"
                        + (" (this rank's matrices)" if dplan is not None else ""),
                "launches": len(tc_ms),
                "avg_launch_ms": (span_ms / per_step) if span_ms else tc_total_ms / len(tc_ms),
                "avg_launch_ms_isolated": tc_total_ms / len(tc_ms),
                "frac_isolated": iso_tflops / peak,
                "stage_avg_ms": {name: statistics.mean(tc_ms[i::3]) for i, name in
                                 enumerate(("gram", "poly", "apply"))},
                "share_of_step": tc_total_ms / ms_prof,
                "timing": ("CUDA events on the launching stream over %d further steps after the "
                           "timed region: one pair around each Newton-Schulz call's run of "
                           "%d launches (avg_launch_ms = span / launches; the launches keep "
                           "their programmatic-dependent-launch overlap, as in the timed "
                           "region), and separately one pair around every launch "
                           "(avg_launch_ms_isolated, stage_avg_ms: each launch then also pays "
                           "its own set-up)" % (reps_tc, int(per_step))) if span_ms else
                          "per-launch CUDA events over %d further steps after the timed region"
                          % reps_tc}
        traffic = read_traffic(wl)
        if traffic is not None and dplan is None:
            roof["traffic"] = traffic
    elif wl.compute == "f32" and (kernel_ms.get("ns_small") or step.whole_call):
        # the fp32 Newton–Schulz: FFMA work against the fp32 CUDA-core peak (the one-launch
        # kernel's own time, else the Newton–Schulz stage's or the whole call's)
        small_ms = kernel_ms.get("ns_small") or st_ns  # per step
        gflop = dense_flops(shapes, wl.steps) / (small_ms / 1000.0) / 1e12
        peak = fp32_peak_tflops(dev)
        roof = {"kernel": "ns_small_kernel" if kernel_ms.get("ns_small") else
                "ns_simt_kernel (timed with the rest of the call)",
                "bound": "alu", "achieved": gflop, "peak": peak,
                "unit": "TFLOP/s", "frac": gflop / peak, "traffic": None,
                "peak_source": "derived: SMs x 128 fp32 FMA lanes x 2 flops x max SM clock",
                "work": "dense flops 4m^2n + 2m^3 per iteration", "avg_launch_ms": small_ms,
                "launches": int(round(len([1 for _, t in tagged if t == "ns_small"]) / reps_tc)),
                "note": ("one cluster of 8 CTAs per matrix: a latency-bound launch on %d of "
                         "the GPU's SMs" % (8 * len(shapes))) if kernel_ms.get("ns_small") else
                        "64x64 FFMA tiles, one launch per product"}
    else:
        mom_b, upd_b = stage_bytes(wl, step)
        gbs = (mom_b + (upd_b or 0)) / ((st_mom + (st_upd if upd_b else 0)) / 1000.0) / 1e9
        roof = {"kernel": "elementwise stages", "bound": "hbm", "achieved": gbs, "peak": hbm,
                "unit": "GB/s", "frac": gbs / hbm, "traffic": None,
                "peak_source": "%s hbm_gbs" % peak_src}
    if step.whole_call:
        stages = {"whole_step": st_step, "ns_tc_launches": st_ns}
        ew_gbs = {"momentum": None, "update": None, "peak": hbm,
                  "fused": "momentum in the staging pass, update in the last product"
                  if step.fused else "one call for the whole step; no per-stage split"
                  if step.fused_sign else
                  "one call per stage and the exchange; no per-stage split"}
    else:
        mom_b, upd_b = stage_bytes(wl, step)
        stages = {"momentum": st_mom, "ns": st_ns, "update": st_upd}
        ew_gbs = {"momentum": mom_b / (st_mom / 1000.0) / 1e9,
                  "update": upd_b / (st_upd / 1000.0) / 1e9 if upd_b else None, "peak": hbm}
    if step.fused:
        launch["call"] = "muon_step (momentum, Newton-Schulz and update in one call)"
    if step.fused_sign:
        launch["call"] = ("sign_muon_step (momentum, Newton-Schulz with packed signs, vote and "
                          "update in one call)")
    if dplan is not None:
        launch["exchange"] = ("all-gather(v) of updated weights" if wl.kind == "muon" else
                              "all-gather of packed signs" if opts.variant == "bits" else
                              "int8 SUM all-reduce")
    line = {
        "metric": metric_name(wl), "value": value, "unit": "steps/s", "n_gpus": world,
        "steps": K, "warmup": Wu, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": scaling, "vs_baseline": None, "dtype": wl.compute, "data": "synthetic",
        "config": cfg, "step": launch,
        "ns_tflops_dense": dense / (st_ns / 1000.0) / 1e12,
        "ns_tflops_alg": alg / (st_ns / 1000.0) / 1e12,
        "stages_ms": stages,
        "elementwise_gbs": ew_gbs,
        "roofline": roof,
        "gpu_launches": launches,
        "clocks": clk,
    }
    return line, step


def per_config_runs(args, dev, local, barrier, max_over_ranks):
    """The other workloads, each measured alone on this GPU (no e2e or CPU baseline)."""
    import torch
    from matrix_aware_optimizers_gb300 import workloads
    out = {}
    opts = parse_args([])  # defaults: 1-bit aggregation, eager, the one-call Muon step
    for c, (K, Wu) in PER_CONFIG.items():
        wl = workloads.workload(c)
        try:
            line, step = measure(opts, wl, dev, 1, 0, local, None, K, Wu, barrier, max_over_ranks)
        except Exception as e:  # report, keep the default line
            out[str(c)] = {"workload": wl.name, "error": "%s: %s" % (type(e).__name__, e)}
            continue
        finally:
            gc.collect()
            torch.cuda.empty_cache()
        r = line["roofline"]
        out[str(c)] = {
            "workload": wl.name, "metric": line["metric"], "value": line["value"],
            "unit": "steps/s", "steps": K, "warmup": Wu, "ms_per_step": line["ms_per_step"],
            "ns_tflops_alg": line.get("ns_tflops_alg"),
            "ns_tflops_dense": line.get("ns_tflops_dense"),
            "roofline": {k: r.get(k) for k in ("kernel", "bound", "achieved", "peak", "unit",
                                               "frac", "frac_isolated", "peak_source",
                                               "avg_launch_ms", "avg_launch_ms_isolated",
                                               "tc_tflops", "tc_share_of_step")
                         if k in r},
            "stages_ms": line["stages_ms"], "gpu_launches": line["gpu_launches"],
            **({"kernels_ms_per_step": line["kernels_ms_per_step"]}
               if "kernels_ms_per_step" in line else {}),
            "clocks": line["clocks"], "parity": PARITY_TESTS[c],
        }
        del step, line
        gc.collect()
        torch.cuda.empty_cache()
    return out


def main():
    args = parse_args()
    from matrix_aware_optimizers_gb300 import workloads
    wl = workloads.workload(args.config)
    if args.compute is not None and args.compute != wl.compute:
        import dataclasses
        if wl.kind == "dion":
            sys.exit("--compute applies to the Muon and Sign-Muon workloads")
        wl = dataclasses.replace(wl, compute=args.compute)
    block = None
    if args.block:
        block = tuple(int(v) for v in args.block.lower().split("x"))
        if wl.kind != "muon" or len(block) != 2 or min(block) < 1:
            sys.exit("--block ROWSxCOLS applies to the Muon workloads (--config 2, 4 or 5)")
    if wl.kind != "sign" and (args.variant != "bits" or args.post_polar):
        sys.exit("--variant / --post-polar apply to the Sign-Muon workloads (--config 1 or 3)")
    if args.impl == "reference":
        run_reference(args, wl, block)
        return

    import torch
    import torch.distributed as dist
    import matrix_aware_optimizers_gb300 as mao

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    mao.lib()
    if args.sweep_hbm:
        if rank == 0:
            sweep_hbm(dev)
        return

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(x):
        return reduce_max(x, dev, world)

    K = args.steps if args.steps is not None else DEFAULT_STEPS[wl.index]
    Wu = max(3, args.warmup if args.warmup is not None else DEFAULT_WARMUP[wl.index])
    line, step = measure(args, wl, dev, world, rank, local, block, K, Wu, barrier,
                         max_over_ranks)
    line = finish_line(args, line, wl, step, K, world, rank, dev, barrier, max_over_ranks)
    default_run = args.config == 2 and block is None and not args.graph and not args.unfused
    if world == 1 and default_run and not args.no_per_config:
        del step
        gc.collect()
        torch.cuda.empty_cache()
        line["per_config"] = per_config_runs(args, dev, local, barrier, max_over_ranks)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def dion_line(wl, step, K, Wu, world, value, ms_step, reps_tc, ms_prof, st_step, tc_ms, launches,
              clk, peaks, peak_src, cfg, scaling, kernel_ms=None):
    """Bench line of a Dion workload: the step is HBM-bound (every matrix element is read and
    written a fixed number of times, 8 m n r flops against about 10 bytes per element)."""
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    need = dion_min_bytes(step)
    gbs = need / (st_step / 1000.0) / 1e9
    flops = sum(8 * w.shape[0] * w.shape[1] * wl.rank for w in step.W)
    tc_total = sum(tc_ms)
    roof = {"kernel": "dion_step (all kernels of one call)", "bound": "hbm", "achieved": gbs,
            "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "traffic": None,
            "peak_source": "%s hbm_gbs" % peak_src,
            "work": "bytes a step must move: X, M, G, Q read; X, M, Q written",
            "tc_launches": len(tc_ms),
            "tc_share_of_step": tc_total / ms_prof if tc_ms else None,
            "tc_tflops": flops * reps_tc / (tc_total / 1000.0) / 1e12 if tc_ms else None}
    return {
        "metric": metric_name(wl), "value": value, "unit": "steps/s", "n_gpus": world,
        "steps": K, "warmup": Wu, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": scaling, "vs_baseline": None, "dtype": wl.compute, "data": "synthetic",
        "config": cfg, "stages_ms": {"dion_step": st_step}, "roofline": roof,
        "kernels_ms_per_step": {k: round(v, 4) for k, v in (kernel_ms or {}).items()},
        "gpu_launches": launches, "clocks": clk,
    }


def finish_line(args, line, wl, step, K, world, rank, dev, barrier, max_over_ranks):
    """Adds the end-to-end leg and (one GPU, rank 0) the oracle's CPU baseline to `line`."""
    from matrix_aware_optimizers_gb300 import workloads
    # ---------------- end to end: host gradients in, host weights out, every step
    if not args.no_e2e:
        if step.dplan is not None:
            line["e2e"] = run_e2e_dist(step, K, dev, barrier, max_over_ranks)
        else:
            line["e2e"] = run_e2e(step, K, world, dev, barrier, max_over_ranks, line["scaling"],
                                  warmup=max(3, args.warmup))

    # ---------------- CPU baseline: the oracle on a bounded sample (rank 0, N = 1)
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        host = host_copy(workloads.generate(
            wl, "cpu", shapes=None if wl.index != 4 else
            [(4096, 4096)] * 4 + [(4096, 14336), (14336, 4096), (4096, 14336)]))
        frac, secs, desc = oracle_sample(wl, host, args.cpu_seconds, variant=args.variant,
                                         post_polar=args.post_polar, block=step.block)
        line["cpu_baseline"] = {"value": frac / secs, "unit": "steps/s", "cores": blas_threads(),
                                "kind": "oracle", "sample": desc + ", %.1f s" % secs}
    return line


def _slab(tensors, device, pin=False):
    """One contiguous buffer holding every tensor (each start 128-byte aligned) and views of
    it shaped like the tensors; returns (buffer, views). Host buffers are pinned."""
    import torch
    dt = tensors[0].dtype
    offs, n = [], 0
    for t in tensors:
        offs.append(n)
        n += (t.numel() + 63) // 64 * 64
    buf = torch.zeros(n, dtype=dt, device=device)
    if pin:
        buf = buf.pin_memory()
    views = [buf[o:o + t.numel()].view(t.shape) for o, t in zip(offs, tensors)]
    for v, t in zip(views, tensors):
        v.copy_(t)
    return buf, views


def _copy_only(K, G_host, G_dsts, W_host, W_srcs, world, scaling, max_over_ranks):
    """The host link alone: the step's K copies each way (gradient slab in, weight slab out)
    on two streams at once, with no compute; an e2e figure cannot exceed this rate."""
    import torch
    main = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    c0.record(main)
    s_in.wait_stream(main)
    s_out.wait_stream(main)
    for k in range(K):
        with torch.cuda.stream(s_in):
            G_dsts[k % len(G_dsts)].copy_(G_host, non_blocking=True)
        with torch.cuda.stream(s_out):
            W_host.copy_(W_srcs[k % len(W_srcs)], non_blocking=True)
    main.wait_stream(s_in)
    main.wait_stream(s_out)
    c1.record(main)
    torch.cuda.synchronize()
    ms_copy = max_over_ranks(c0.elapsed_time(c1))
    h2d = G_host.numel() * G_host.element_size()
    d2h = W_host.numel() * W_host.element_size()
    return {"value": job_throughput(ms_copy, K, world, scaling),
            "h2d_gbs": h2d * K / (ms_copy / 1000.0) / 1e9,
            "d2h_gbs": d2h * K / (ms_copy / 1000.0) / 1e9,
            "note": "the step's copies alone, both directions at once: the host-link bound "
                    "of the e2e figure"}


def run_e2e(step, K, world, dev, barrier, max_over_ranks, scaling="strong", warmup=3):
    """The same step with host data: every step copies its gradients from pinned host memory
    (one copy of one contiguous slab) and reads the updated weights back (one copy). The
    first `warmup` steps of the sequence are run untimed; K are timed.

    Copies run on their own streams and overlap other work where the data allow it: the
    gradients of step k+1 go into the second of two device slabs while step k computes, and
    the weights of step k are read back while step k+1 runs its momentum and Newton–Schulz
    stages (its update waits for that read). A one-call step (muon_step, or dion_step) reads
    W from one of two device slabs and writes the new W into the other (its W_out / X_out),
    so the read-back of step k's weights overlaps step k+1, which writes the slab step k
    read. Every step still moves all of its bytes.
    """
    import torch
    main = torch.cuda.current_stream()
    if any(g.dtype != step.G[0].dtype for g in step.G) or any(w.dtype != step.W[0].dtype for w in step.W):
        raise ValueError("one dtype per slab")
    G_host, _ = _slab([g.cpu() for g in step.G], "cpu", pin=True)
    W_host, _ = _slab([w.cpu() for w in step.W], "cpu", pin=True)
    G_dev = [_slab(step.G, dev) for _ in range(2)]
    W_dev, W_views = _slab(step.W, dev)
    G_orig, W_orig = step.G, step.W
    step.W = W_views
    dion = step.wl.kind == "dion"
    fused = getattr(step, "fused", False) or dion  # one call updates W: muon_step, dion_step
    # fused: two weight slabs, read one and write the other; one read-back event per slab
    W_bufs = [(W_dev, W_views)] + ([_slab(step.W, dev)] if fused else [])
    w_read_slab = [torch.cuda.Event() for _ in W_bufs]
    h2d = G_host.numel() * G_host.element_size()
    d2h = W_host.numel() * W_host.element_size()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    g_free = [torch.cuda.Event() for _ in range(2)]
    g_ready = [torch.cuda.Event() for _ in range(2)]
    w_done, w_read = torch.cuda.Event(), torch.cuda.Event()
    for ev in g_free:
        ev.record(main)
    w_read.record(main)
    for ev in w_read_slab:
        ev.record(main)
    W_src = W_dev
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    host_call = getattr(step, "fused", False) and not dion
    if host_call:
        # one muon_step_host call per step (host gradients in, host weights out, through the
        # C ABI), rotating over n streams with n gradient slabs, n weight slabs and n host
        # weight buffers: step k reads weight slab k % n and writes slab (k + 1) % n, and
        # waits for step k-1's compute event; everything else a step touches was last used
        # on its own stream, so each step's copies overlap its neighbours' compute
        wl = step.wl
        n = 3 if h2d <= (4 << 30) else 2
        streams = [torch.cuda.Stream() for _ in range(n)]
        done = [torch.cuda.Event() for _ in range(n)]
        Gs = [G_dev[0], G_dev[1]] + [_slab(G_orig, dev) for _ in range(n - 2)]
        Ws = [W_bufs[0], W_bufs[1]] + [_slab(W_orig, dev) for _ in range(n - 2)]
        W_hosts = [W_host] + [_slab([w.cpu() for w in W_orig], "cpu", pin=True)[0]
                              for _ in range(n - 1)]
        for st_, ev in zip(streams, done):
            ev.record(st_)
        torch.cuda.synchronize()

        def host_steps(k0, k1):
            for st_ in streams:
                st_.wait_stream(main)
            for k in range(k0, k1):
                b = k % n
                step.mao.muon_step_host(
                    Ws[b][1], step.M, Gs[b][1], wl.mu, wl.lr, G_host, Gs[b][0], W_hosts[b],
                    Ws[(k + 1) % n][0], wl.steps, wl.coeffs, wl.eps, wl.compute, ws=step.ws,
                    W_out=Ws[(k + 1) % n][1], stream=streams[b],
                    wait_event=done[(k - 1) % n] if k > 0 else None, record_event=done[b])
            for st_ in streams:
                main.wait_stream(st_)

        host_steps(0, warmup)
        torch.cuda.synchronize()
        barrier()
        e0.record(main)
        host_steps(warmup, warmup + K)
        e1.record(main)
        torch.cuda.synchronize()
        barrier()
        ms = max_over_ranks(e0.elapsed_time(e1))
        for w, v in zip(W_orig, Ws[(warmup + K) % n][1]):
            w.copy_(v)
        step.G, step.W = G_orig, W_orig
        copy_only = _copy_only(K, G_host, [g[0] for g in Gs], W_host, [w[0] for w in Ws], world,
                               scaling, max_over_ranks)
        return {"value": job_throughput(ms, K, world, scaling), "unit": "steps/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K,
                "copy_only": copy_only,
                "call": "muon_step_host (C ABI: host gradients in, host weights out)",
                "copies": "one pinned H2D slab and one D2H slab per step inside each call; %d "
                          "streams in rotation, step k waiting on step k-1's compute event" % n}
    def steps(k0, k1):
        for k in range(k0, k1):
            one_step(k)

    def one_step(k):
        nonlocal W_src
        b = k % 2
        s_in.wait_event(g_free[b])            # step k-2 has read this slab
        with torch.cuda.stream(s_in):
            G_dev[b][0].copy_(G_host, non_blocking=True)
        g_ready[b].record(s_in)
        main.wait_event(g_ready[b])
        step.G = G_dev[b][1]
        if getattr(step, "fused_sign", False):
            main.wait_event(w_read)           # the previous read-back of W is complete
            step()                            # one sign_muon_step call
            g_free[b].record(main)
        elif not fused:
            step.momentum()
            g_free[b].record(main)
            step.ns()
            main.wait_event(w_read)           # the previous read-back of W is complete
            step.update()
        else:
            src, dst = k % 2, 1 - k % 2
            step.W = W_bufs[src][1]
            main.wait_event(w_read_slab[dst])  # step k-2's weights have been read back
            step.fused_call(W_out=W_bufs[dst][1])
            g_free[b].record(main)
            W_src = W_bufs[dst][0]
        w_done.record(main)
        s_out.wait_event(w_done)
        with torch.cuda.stream(s_out):
            W_host.copy_(W_src, non_blocking=True)
        w_read.record(s_out)
        if fused:
            w_read_slab[1 - k % 2].record(s_out)

    steps(0, warmup)
    main.wait_event(w_read)
    torch.cuda.synchronize()
    barrier()
    e0.record(main)
    steps(warmup, warmup + K)
    main.wait_event(w_read)
    e1.record(main)
    torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1))
    last_views = W_bufs[(warmup + K) % 2][1] if fused else W_views
    step.G, step.W = G_orig, W_orig
    for w, v in zip(W_orig, last_views):
        w.copy_(v)
    copy_only = _copy_only(K, G_host, [g[0] for g in G_dev], W_host, [w[0] for w in W_bufs], world,
                           scaling, max_over_ranks)
    return {"value": job_throughput(ms, K, world, scaling), "unit": "steps/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": K,
            "copy_only": copy_only,
            "copies": "one pinned H2D slab and one D2H slab per step, on copy streams overlapping "
                      "the neighbouring steps' compute" +
                      ("; two device weight slabs, read one, write the other (%s)"
                       % ("dion_step's X_out" if dion else "muon_step's W_out") if fused else "")}


def run_e2e_dist(step, K, dev, barrier, max_over_ranks):
    """End to end across ranks: every step, each rank copies its share of the gradients in
    from pinned host memory (the matrices it owns, or its workers' gradients) and reads its
    result back (the weights it updated; Sign-Muon: the new W), around the step and its
    exchange. Copies and compute run in order on the step's stream."""
    import torch
    main = torch.cuda.current_stream()
    G_host, _ = _slab([g.cpu() for g in step.G], "cpu", pin=True)
    G_dev, G_views = _slab(step.G, dev)
    G_orig = step.G
    step.G = G_views
    if step.wl.kind == "muon":
        out_dev = step.dplan.layout.segment(step.flat, step.dplan.rank)
    else:
        out_dev = step.W[0].view(-1)
    out_host = torch.empty(out_dev.shape, dtype=out_dev.dtype).pin_memory()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for _ in range(K):
        G_dev.copy_(G_host, non_blocking=True)
        step()
        out_host.copy_(out_dev, non_blocking=True)
    e1.record(main)
    torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1))
    step.G = G_orig
    return {"value": job_throughput(ms, K, step.dplan.world, "strong"), "unit": "steps/s",
            "h2d_bytes_per_step": G_host.numel() * G_host.element_size(),
            "d2h_bytes_per_step": out_host.numel() * out_host.element_size(), "steps": K,
            "copies": "rank 0's figures: its gradient slab in, its updated weights out, in "
                      "stream order with the step"}


def read_traffic(wl):
    """DRAM bytes per launch of the tensor-core kernel from the committed ncu summary of this
    workload, or None when that summary was taken on a different kernel source."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "ns_tc_kernel_%s.md" % wl.name)
    src = os.path.join(ROOT, "matrix_aware_optimizers_gb300", "csrc", "ns_tc.cu")
    try:
        with open(src, "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()[:16]
        traffic, srchash = None, None
        with open(path) as f:
            for line in f:
                if line.startswith("traffic_bytes_per_launch:"):
                    traffic = float(line.split(":", 1)[1])
                if line.startswith("kernel_source_sha256_16:"):
                    srchash = line.split(":", 1)[1].strip()
        if traffic is not None and srchash == digest:
            return traffic
    except OSError:
        pass
    return None


if __name__ == "__main__":
    main()
