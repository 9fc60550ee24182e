"""Benchmark: QuantSpec decode attention over the hierarchical quantized KV
cache on one GB300 (replicas over N GPUs, no collective on the data path).

One step = one speculative round (gamma = 4) of the whole hot path on the
Llama-2-7B-shaped 32k workload (batch 1, 32 heads, head_dim 128, G = 128,
starting at 254 quantized groups + a full 256-token fp16 buffer = 32,768
tokens):
    need_flush + quantize-on-flush (128 tokens x 32 heads),
    4 x (append 1 draft token + draft decode attention, 1 query, C_U only),
    rollback of the 4 draft tokens, append 5 target tokens,
    verify decode attention (5 queries, INT8), rollback of 4 - a (a seeded),
then the counters are restored to the starting state (a device copy) so every
step does the same work.  ``value`` is algorithmic bytes per step / step time
(GB/s), summed over ranks.  Bytes are counted per sequence from its own
counters (a flush only for the sequences whose mask is set).

Per-call numbers (draft_us, verify_us, flush_us) time one call at a time
(CUDA-graph replay) with the L2 evicted before each call by reading a 256 MB
buffer; the roofline object uses the calls' durations inside the step.  The
``configs`` object reports the other workloads (tiny, 128k, batched 32k,
ragged): the same round on each, with the durations of the attention calls
inside it and the round's own time.
"""
import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/step & HBM GB/s (draft 4-bit / verify 8-bit) at 32k ctx"
GAMMA = 4
KB = 1024
G_TOK = 128
RING = 2 * G_TOK


def kernel_source_hash():
    """sha256 over the attention kernel sources (to tell whether a stored ncu
    traffic figure still describes the kernel that runs)."""
    import hashlib
    h = hashlib.sha256()
    for f in ("qs_attn.cu", "qs_common.cuh"):
        with open(os.path.join(ROOT, "hierarchical_quantized_kv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def stored_traffic(kind):
    """DRAM bytes per launch of the split kernel from the committed ncu
    summary, or None when the kernel changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "split_kernel_traffic_32k.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha256") != kernel_source_hash():
            return None
        return int(kv["%s_dram_bytes_per_launch" % kind])
    except (OSError, KeyError, ValueError):
        return None


def rank_max(dist, world, x, device):
    """x maximized over the ranks: the slowest replica sets the job's time."""
    if world == 1:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(step_bytes_per_rank, world, ms):
    """Whole-job throughput: every replica's bytes per step over the slowest
    replica's step time (weak scaling)."""
    return step_bytes_per_rank * world / (ms * 1e-3) / 1e9


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------- bytes

def attn_bytes(ng, fill, n_q, mode_draft, BH, group=1, upper_bits=4):
    """Algorithmic bytes of one decode-attention call per the method: the
    quantized planes it must read (draft: C_U + scales/zeros = 136 B per
    token-head, or with the two-bit draft C_U2 + scales/zeros = 72 B;
    verify: all 8 bits + scales/zeros = 264 B), the fp16 buffer tokens (512 B
    each), the queries and the outputs (group query heads per KV head)."""
    up = 8 * KB * upper_bits // 4
    grp = (up + up + KB) if mode_draft else (4 * 8 * KB + KB)
    return BH * (ng * grp + fill * 512 + group * n_q * 256 * 2)


FLUSH_BYTES_PER_HEAD = 2 * 128 * 256 + 4 * 8 * KB + KB   # read the oldest half (K, V), write planes + meta


def append_bytes(n, BH):
    return BH * n * 512 * 2


def prefill_bytes(L, BH, G=128):
    """qs_prefill of an L-token prompt: read K and V, write the groups
    (both planes + meta, 33,792 B per group-head) and the buffer tokens."""
    ng = 0 if L <= 2 * G else -(-(L - 2 * G) // G)
    return BH * (L * 512 + ng * 33792 + (L - ng * G) * 512)


def round_plan(ng0, f0, H, gamma=GAMMA, upper_bits=4):
    """The counters of every sequence through one speculative round and the
    algorithmic bytes of each call, counted per sequence: the flush only for
    sequences whose buffer cannot take the gamma + 1 target tokens
    (fill + gamma + 1 > 2G), then gamma drafts over fill1 + 1 .. fill1 + gamma
    buffered tokens and a (gamma + 1)-query verify over fill1 + gamma + 1."""
    ng0 = np.asarray(ng0, np.int64)
    f0 = np.asarray(f0, np.int64)
    B = len(ng0)
    mask = (f0 + gamma + 1 > RING).astype(np.int64)
    ng1 = ng0 + mask
    f1 = f0 - G_TOK * mask
    draft = [int(sum(attn_bytes(int(n), int(f) + i + 1, 1, True, H, upper_bits=upper_bits)
                     for n, f in zip(ng1, f1))) for i in range(gamma)]
    verify = int(sum(attn_bytes(int(n), int(f) + gamma + 1, gamma + 1, False, H)
                     for n, f in zip(ng1, f1)))
    b = {"flush": FLUSH_BYTES_PER_HEAD * H * int(mask.sum()), "draft": draft, "verify": verify,
         "append": append_bytes(gamma, B * H) + append_bytes(gamma + 1, B * H)}
    step = b["flush"] + sum(b["draft"]) + b["verify"] + b["append"]
    return {"mask": mask, "ng1": ng1, "f1": f1, "bytes": b, "step": step}


# --------------------------------------------------------------- clocks

# NVML clock-event reason bits (read-only queries)
_REASONS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8 | 0x80), ("sw_thermal_slowdown", 0x20),
            ("hw_thermal_slowdown", 0x40))


def nvml_reader(torch=None, index=0):
    """A callable returning (sm_mhz, sm_max_mhz, power_w, reasons) for the
    benchmark's GPU through NVML's read-only queries, or None when NVML is not
    available.  The device is found by its UUID (CUDA and NVML may number
    devices differently), else by index."""
    try:
        nv = ctypes.CDLL("libnvidia-ml.so.1")
    except OSError:
        return None
    try:
        if nv.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        ok = False
        if torch is not None:
            try:
                uuid = str(torch.cuda.get_device_properties(index).uuid)
                uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
                ok = nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
            except Exception:
                ok = False
        if not ok and nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) != 0:
            return None
        try:
            reasons_fn = nv.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            reasons_fn = nv.nvmlDeviceGetCurrentClocksThrottleReasons
        smax = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(smax)) != 0:
            return None
    except Exception:
        return None

    def read():
        sm, mw, bits = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) != 0:
            return None
        power = mw.value / 1e3 if nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0 else None
        reasons = frozenset()
        if reasons_fn(h, ctypes.byref(bits)) == 0:
            reasons = frozenset(n for n, m in _REASONS if bits.value & m)
        return float(sm.value), float(smax.value), power, reasons
    return read


class ClockSampler:
    """SM clock, power and throttle reasons sampled during the timed region.

    With a reader (NVML) a thread samples every ``period_s`` (1 ms), so even a
    few-millisecond timed region holds several samples; without one it falls
    back to ``nvidia-smi -lms 100``.  Samples are (host time, sm_mhz,
    sm_max_mhz, power_w, reasons)."""

    def __init__(self, reader=None, period_s=0.001, smi_index=None):
        self.samples = []
        self.proc = None
        self.thread = None
        self._halt = threading.Event()
        self.source = None
        if reader is not None:
            self.source = "nvml %.0f ms" % (period_s * 1e3)

            def loop():
                while not self._halt.is_set():
                    s = reader()
                    if s is not None:
                        self.samples.append((time.time(),) + tuple(s))
                    time.sleep(period_s)
            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
        elif smi_index is not None:
            self.source = "nvidia-smi 100 ms"
            fields = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                      "clocks_event_reasons.hw_thermal_slowdown,"
                      "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(smi_index), "--query-gpu=" + fields,
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception:
                self.proc = None
                return
            self.thread = threading.Thread(target=self._read_smi, daemon=True)
            self.thread.start()

    @classmethod
    def from_samples(cls, samples):
        """A sampler holding the given samples (no thread, no process)."""
        s = cls()
        s.samples = list(samples)
        return s

    @staticmethod
    def parse_smi(line):
        """One nvidia-smi CSV line -> (sm, sm_max, power, reasons), None where
        a field does not parse."""
        p = [x.strip() for x in line.split(",")]
        if len(p) < 7:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = frozenset(n for n, v in zip(names, p[3:7]) if v.lower().startswith("active"))
        return num(p[0]), num(p[1]), num(p[2]), reasons

    def _read_smi(self):
        for line in self.proc.stdout:
            s = self.parse_smi(line)
            if s is not None:
                self.samples.append((time.time(),) + s)

    def stop(self):
        self._halt.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def count(self, t0, t1):
        return sum(1 for s in list(self.samples) if t0 <= s[0] <= t1)

    def summary(self, t0, t1, note="inside timed region"):
        inside = [s for s in list(self.samples) if t0 <= s[0] <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [s[1] for s in inside if s[1] is not None]
        smax = [s[2] for s in inside if s[2] is not None]
        power = [s[3] for s in inside if s[3] is not None]
        reasons = set()
        for s in inside:
            reasons |= set(s[4])
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
               "power_w_max": max(power) if power else None, "samples": len(inside),
               "note": note}
        if self.source:
            out["source"] = self.source
        return out


# ------------------------------------------------------------ native arm

def kv_tokens_parallel(synthetic, w, b, n, pool):
    """synthetic.kv_tokens(w, b, 0, n), its 128-token chunks drawn in parallel
    (each chunk has its own seeded generator, so the values are the same)."""
    k = np.empty((w.H, n, w.D), np.float16)
    v = np.empty_like(k)

    def one(c):
        m = min(synthetic.CHUNK, n - c * synthetic.CHUNK)
        kc, vc = synthetic.kv_chunk(w, b, c, m)
        k[:, c * synthetic.CHUNK:c * synthetic.CHUNK + m] = kc
        v[:, c * synthetic.CHUNK:c * synthetic.CHUNK + m] = vc
    list(pool.map(one, range(-(-n // synthetic.CHUNK))))
    return k, v


def fast_prefill(torch, qs, synthetic, cache, w):
    """Bring ``cache`` to the workload's starting state (its n_groups and
    fill per sequence) in a few public calls: qs_prefill of each sequence's
    quantized tokens (which leaves the last 2G of them in the buffer), two
    masked flushes that quantize those, one append of the buffer tokens and a
    rollback that drops the padding and commits the rest.  The groups are the
    consecutive G-token chunks of the stream either way, so the state equals
    the one appending the whole context token by token would leave."""
    dev = cache.state.device
    B, H, D, G = w.B, w.H, w.D, w.G
    tq = np.array(w.quantized, np.int64)
    f = np.array(w.fill, np.int64)
    assert np.all(tq % G == 0) and np.all((f >= 0) & (f <= 2 * G))
    qs.qs_state_reset(cache)
    with ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1))) as pool:
        tmax = int(tq.max(initial=0))
        if tmax:
            kd = torch.zeros((B, H, tmax, D), dtype=torch.float16, device=dev)
            vd = torch.zeros_like(kd)
            for b in range(B):
                if tq[b]:
                    k, v = kv_tokens_parallel(synthetic, w, b, int(tq[b]), pool)
                    kd[b, :, :tq[b]].copy_(torch.from_numpy(k))
                    vd[b, :, :tq[b]].copy_(torch.from_numpy(v))
            qs.qs_prefill(cache, kd, vd, torch.from_numpy(tq.astype(np.int32)).to(dev))
            del kd, vd
            for k_ in range(2):
                mask = torch.from_numpy((tq >= G * (k_ + 1)).astype(np.uint8)).to(dev)
                qs.qs_quantize_flush(cache, mask)
        fmax = int(f.max(initial=0))
        if fmax:
            kb = np.zeros((B, H, fmax, D), np.float16)
            vb = np.zeros_like(kb)
            for b in range(B):
                if f[b]:
                    kb[b, :, :f[b]], vb[b, :, :f[b]] = synthetic.kv_tokens(w, b, int(tq[b]),
                                                                          int(f[b]))
            qs.qs_buffer_append(cache, torch.from_numpy(kb).to(dev), torch.from_numpy(vb).to(dev))
            qs.qs_buffer_rollback(cache, torch.from_numpy((fmax - f).astype(np.int32)).to(dev))
    st = cache.state.cpu().numpy()
    assert np.array_equal(st[:, 0], tq // G) and np.array_equal(st[:, 1], f), st[:, :5]
    assert np.all(qs.qs_get_errors(cache) == 0)


class Round:
    """Device state and inputs of the benchmark step on one GPU."""

    def __init__(self, torch, w, seed, upper_bits=4, fused=True):
        """fused: the flush decides its own mask (qs_quantize_flush_due) and
        each attention call takes its appended tokens in the same launch
        (qs_attn_decode_append); else qs_need_flush, qs_quantize_flush and
        separate qs_buffer_append calls."""
        from hierarchical_quantized_kv_gb300 import qs, synthetic
        self.torch, self.qs, self.w = torch, qs, w
        self.fused = fused
        dev = torch.device("cuda")
        B, H, D = w.B, w.H, w.D
        self.cache = qs.Cache(B, H, max(w.n_groups) + 2, upper_bits=upper_bits)
        fast_prefill(torch, qs, synthetic, self.cache, w)
        torch.cuda.synchronize()
        self.state0 = self.cache.state.clone()
        rng = np.random.default_rng([seed, 77])
        f16 = lambda *s: torch.from_numpy(rng.standard_normal(s).astype(np.float16)).to(dev)
        self.kd = [f16(B, H, 1, D) for _ in range(GAMMA)]
        self.vd = [f16(B, H, 1, D) for _ in range(GAMMA)]
        self.kt, self.vt = f16(B, H, GAMMA + 1, D), f16(B, H, GAMMA + 1, D)
        self.qd = [torch.from_numpy(synthetic.queries(w, i, 1)).to(dev) for i in range(GAMMA)]
        self.qv = torch.from_numpy(synthetic.queries(w, GAMMA, GAMMA + 1)).to(dev)
        self.od = [torch.empty_like(q) for q in self.qd]
        self.ov = torch.empty_like(self.qv)
        self.lse = torch.empty((B, H, GAMMA + 1), dtype=torch.float32, device=dev)

        # The step's inputs live in one device buffer and its outputs in
        # another (views at 16-byte aligned offsets), so the end-to-end run
        # moves each with a single copy.
        def arena(tensors):
            sizes = [t.numel() * t.element_size() for t in tensors]
            offs, o = [], 0
            for n in sizes:
                offs.append(o)
                o += -(-n // 16) * 16
            buf = torch.empty(o, dtype=torch.uint8, device=dev)
            views = []
            for t, off, n in zip(tensors, offs, sizes):
                v = buf[off:off + n].view(t.dtype).view(t.shape)
                v.copy_(t)
                views.append(v)
            return buf, views
        self.in_arena, v = arena(self.kd + self.vd + [self.kt, self.vt] + self.qd + [self.qv])
        self.kd, self.vd = v[:GAMMA], v[GAMMA:2 * GAMMA]
        self.kt, self.vt = v[2 * GAMMA], v[2 * GAMMA + 1]
        self.qd, self.qv = v[2 * GAMMA + 2:3 * GAMMA + 2], v[3 * GAMMA + 2]
        self.out_arena, v = arena(self.od + [self.ov, self.lse])
        self.od, self.ov, self.lse = v[:GAMMA], v[GAMMA], v[GAMMA + 1]
        n_ws = max(qs.qs_attn_workspace_size(self.cache, 1), qs.qs_attn_workspace_size(self.cache, GAMMA + 1))
        self.ws = torch.empty(n_ws, dtype=torch.uint8, device=dev)
        self.mask = torch.zeros(B, dtype=torch.uint8, device=dev)
        self.drop_draft = torch.full((B,), GAMMA, dtype=torch.int32, device=dev)
        self.drops = [torch.from_numpy(GAMMA - synthetic.accepted_counts(w, s)).to(dev) for s in range(16)]
        self.scale = 1.0 / np.sqrt(D)
        st = self.state0.cpu().numpy()
        self.plan = round_plan(st[:, 0], st[:, 1], H, upper_bits=upper_bits)
        # state after the step's flush (per sequence)
        self.ng1, self.f1 = self.plan["ng1"], self.plan["f1"]
        self.bytes = self.plan["bytes"]
        self.step_bytes = self.plan["step"]
        # (need_flush +) flush, GAMMA x (append +) draft, rollback, (append +) verify, rollback
        self.launches_per_step = (1 if fused else 2) + GAMMA * (1 if fused else 2) + 1 + \
            (1 if fused else 2) + 1

    def step(self, s, host=None, ev=None, external=False, extra=None, seq=False):
        """One speculative round.  ev: a list that receives (kind, start, end)
        CUDA events recorded around each attention call (as graph nodes when
        the step is captured with external=True); with seq=True one pair of
        events around the run of gamma draft calls instead (kind
        "draft_seq": consecutive launches keep their overlap).  extra =
        "draft" or "verify": one more such attention call (without an append)
        right after each of that kind, for the marginal in-step time."""
        qs, c = self.qs, self.cache
        torch = self.torch
        if ev is not None:
            ev.clear()

        mk = (lambda: torch.cuda.Event(enable_timing=True, external=True)) if external else \
            (lambda: torch.cuda.Event(enable_timing=True))

        def timed(kind, fn):
            if ev is None or (seq and kind == "draft"):
                return fn()
            e0, e1 = mk(), mk()
            e0.record()
            fn()
            e1.record()
            ev.append((kind, e0, e1))

        if host is not None:
            host.h2d(self)
        if self.fused:  # the sequences that cannot take the gamma + 1 targets flush
            qs.qs_quantize_flush_due(c, GAMMA + 1)
        else:
            qs.qs_need_flush(c, GAMMA + 1, self.mask)
            qs.qs_quantize_flush(c, self.mask)
        if ev is not None and seq:
            s0, s1 = mk(), mk()
            s0.record()
        for i in range(GAMMA):
            if self.fused:  # append the draft token and attend in one launch
                timed("draft", lambda i=i: qs.qs_attn_decode_append(
                    c, qs.QS_DRAFT_UPPER4, self.kd[i], self.vd[i], self.qd[i], self.scale,
                    self.od[i], None, self.ws))
                if extra == "draft":
                    qs.qs_attn_decode(c, qs.QS_DRAFT_UPPER4, self.qd[i], self.scale, self.od[i],
                                      None, self.ws)
            else:
                qs.qs_buffer_append(c, self.kd[i], self.vd[i])
                timed("draft", lambda i=i: qs.qs_attn_decode(c, qs.QS_DRAFT_UPPER4, self.qd[i],
                                                             self.scale, self.od[i], None, self.ws))
        if ev is not None and seq:
            s1.record()
            ev.append(("draft_seq", s0, s1))
        qs.qs_buffer_rollback(c, self.drop_draft)
        if self.fused:
            timed("verify", lambda: qs.qs_attn_decode_append(
                c, qs.QS_VERIFY_INT8, self.kt, self.vt, self.qv, self.scale, self.ov, self.lse,
                self.ws))
            if extra == "verify":
                qs.qs_attn_decode(c, qs.QS_VERIFY_INT8, self.qv, self.scale, self.ov, self.lse,
                                  self.ws)
        else:
            qs.qs_buffer_append(c, self.kt, self.vt)
            timed("verify", lambda: qs.qs_attn_decode(c, qs.QS_VERIFY_INT8, self.qv, self.scale,
                                                      self.ov, self.lse, self.ws))
        qs.qs_buffer_rollback(c, self.drops[s % len(self.drops)])
        c.state.copy_(self.state0)
        if host is not None:
            host.d2h(self)

    # states for single-call timing: per-sequence groups and fill
    def set_state(self, ng, fill):
        torch = self.torch
        st = self.state0.clone()
        st[:, 0] = torch.as_tensor(np.asarray(ng), dtype=torch.int32, device=st.device)
        st[:, 1] = torch.as_tensor(np.asarray(fill), dtype=torch.int32, device=st.device)
        st[:, 2] = 0
        self.cache.state.copy_(st)


class HostIO:
    """Pinned host buffers for the end-to-end number: every step copies its
    inputs host -> device and its outputs device -> host (one copy each: the
    step's inputs and outputs are packed in one device buffer each)."""

    def __init__(self, torch, r):
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu())
        self.ins = [(pin(r.in_arena), r.in_arena)]
        self.outs = [(r.out_arena, torch.empty(r.out_arena.shape, dtype=torch.uint8, pin_memory=True))]
        self.h2d_bytes = sum(h.numel() * h.element_size() for h, _ in self.ins)
        self.d2h_bytes = sum(h.numel() * h.element_size() for _, h in self.outs)

    def h2d(self, r):
        for h, d in self.ins:
            d.copy_(h, non_blocking=True)

    def d2h(self, r):
        for d, h in self.outs:
            h.copy_(d, non_blocking=True)


def capture(torch, fn):
    """fn's launches captured once as a CUDA graph (the calls are stream
    ordered and allocate nothing, so replaying the graph repeats them)."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_calls(torch, fn, setup, iters, l2_scratch):
    """Mean device time of one call (replayed from a CUDA graph) over iters
    calls, L2 flushed before each by reading a buffer twice the L2 size (a
    read leaves no dirty lines for the timed call to write back)."""
    setup()
    g = capture(torch, fn)
    ts = []
    sink = torch.empty((), dtype=l2_scratch.dtype, device=l2_scratch.device)
    for _ in range(iters):
        setup()
        torch.sum(l2_scratch, dim=0, out=sink)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)  # us
    return statistics.mean(ts[1:]) if len(ts) > 1 else ts[0]


def external_events_supported(torch):
    try:
        torch.cuda.Event(enable_timing=True, external=True)
        return True
    except TypeError:
        return False


def in_step_launch_times(torch, r, n_rep):
    """Device time of the attention calls inside the step: the steps are
    captured with CUDA events as graph nodes and replayed n_rep times (eager
    steps with events where torch cannot record events into a graph).
    "draft" and "verify": events around each call.  An event node between
    two launches ends the overlap of the later launch's start with the
    earlier one's end (programmatic dependent launch), so each such figure
    carries a launch latency the timed step does not.  "draft_seq": events
    around the step's run of gamma consecutive draft calls, divided by gamma
    (the launches inside the run keep their overlap, as in the timed step).
    Returns ({kind: [us, ...]}, how)."""
    launch = {"draft": [], "verify": [], "draft_seq": []}
    n_steps = min(4, len(r.drops))  # distinct steps (rollback counts) captured
    n_rep = max(n_rep, 6 * n_steps)
    if external_events_supported(torch):
        recs, graphs = [], []
        for seq in (False, True):
            for s in range(n_steps):
                rec = []
                graphs.append(capture(torch, lambda s=s, rec=rec, seq=seq:
                                      r.step(s, ev=rec, external=True, seq=seq)))
                recs.append(rec)
        for i in range(n_rep):
            k = i % len(graphs)
            graphs[k].replay()
            torch.cuda.synchronize()
            if i >= len(graphs):
                for kind, e0, e1 in recs[k]:
                    t = e0.elapsed_time(e1) * 1e3
                    launch[kind].append(t / GAMMA if kind == "draft_seq" else t)
        how = ("CUDA events captured as graph nodes, %d graph-replayed steps after the timed region"
               % (n_rep - len(graphs)))
    else:
        recs = []
        for s in range(n_rep):
            rec = []
            r.step(s, ev=rec, seq=bool(s & 1))
            recs.append(rec)
        torch.cuda.synchronize()
        for rec in recs[2:]:
            for kind, e0, e1 in rec:
                t = e0.elapsed_time(e1) * 1e3
                launch[kind].append(t / GAMMA if kind == "draft_seq" else t)
        how = "CUDA events in %d eager steps" % (n_rep - 2)
    r.cache.state.copy_(r.state0)
    return launch, how


def marginal_us(torch, r, kind, base_graphs, n, rounds=3):
    """Marginal device time of one attention call of `kind` inside the step
    (programmatic dependent launch overlap included): the step's graphs and
    the same step with one more such call after each one, replayed n times
    each, alternately; the least difference of the per-step times over the
    rounds, per added call."""
    extra = [capture(torch, lambda s=s: r.step(s, extra=kind)) for s in range(len(r.drops))]
    per_step = GAMMA if kind == "draft" else 1
    diffs = []
    for _ in range(rounds):
        a = replay_us(torch, base_graphs, n)
        b = replay_us(torch, extra, n)
        diffs.append((b - a) / per_step)
    r.cache.state.copy_(r.state0)
    return min(diffs)


def replay_us(torch, graphs, n):
    """Mean device time per replay of the step graphs, n replays in a row."""
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for s in range(n):
        graphs[s % len(graphs)].replay()
    b.record()
    b.synchronize()
    return a.elapsed_time(b) / n * 1e3


def config_round(torch, qs, synthetic, name, peak, n_rep=40, n_replay=100):
    """The speculative round on another workload: the attention calls'
    durations inside the round (CUDA events) with their algorithmic bytes,
    GB/s and fraction of the HBM peak, and the round's own time by graph
    replay.  Bytes per sequence from its own counters."""
    w = synthetic.CONFIGS[name]()
    t_setup = time.perf_counter()
    r = Round(torch, w, seed=0)
    setup_s = time.perf_counter() - t_setup
    for s in range(3):
        r.step(s)
    torch.cuda.synchronize()
    launch, how = in_step_launch_times(torch, r, n_rep)
    graphs = [capture(torch, lambda s=s: r.step(s)) for s in range(len(r.drops))]
    replay_us(torch, graphs, 10)
    round_us = replay_us(torch, graphs, n_replay)
    errs = qs.qs_get_errors(r.cache)
    assert np.all(errs == 0), errs
    d_us, v_us = float(np.mean(launch["draft_seq"])), float(np.mean(launch["verify"]))
    d_call_us = float(np.mean(launch["draft"]))
    d_b = float(np.mean(r.bytes["draft"]))
    v_b = r.bytes["verify"]
    ctx = np.array(w.context)
    out = {
        "workload": w.name, "B": w.B, "H": w.H,
        "context": int(ctx[0]) if len(set(ctx)) == 1 else
        {"min": int(ctx.min()), "max": int(ctx.max()), "mean": round(float(ctx.mean()), 1)},
        "fill": int(w.fill[0]) if len(set(w.fill)) == 1 else
        {"min": int(min(w.fill)), "max": int(max(w.fill))},
        "flushing_sequences": int(r.plan["mask"].sum()),
        "draft_us": round(d_us, 2), "draft_bytes": int(d_b), "draft_gbs": round(d_b / d_us / 1e3, 1),
        "draft_us_events_per_call": round(d_call_us, 2),
        "verify_us": round(v_us, 2), "verify_bytes": int(v_b),
        "verify_gbs": round(v_b / v_us / 1e3, 1),
        "round_us": round(round_us, 2), "round_bytes": int(r.step_bytes),
        "round_gbs": round(r.step_bytes / round_us / 1e3, 1),
        "launch_timing": how + "; draft: events around the run of %d draft calls, per call; "
                               "verify: events around the call" % GAMMA,
        "setup_s": round(setup_s, 1)}
    if d_b > 2 * 129e6:  # working set larger than L2: an HBM roofline figure
        out["draft_frac"] = round(d_b / d_us / 1e3 / peak, 4)
        out["verify_frac"] = round(v_b / v_us / 1e3 / peak, 4)
    else:
        out["note"] = "working set fits in L2; no HBM roofline figure"
    del graphs, r
    torch.cuda.empty_cache()
    return out


def two_bit_calls(torch, qs, synthetic, w, l2, it):
    """The two-bit draft layout (upper_bits 2: the draft reads the top two
    bits of each code) on the benchmark workload: per-call draft and 5-query
    verify times and GB/s, L2 evicted before each call."""
    r = Round(torch, w, seed=1, upper_bits=2)
    res = {"workload": w.name, "upper_bits": 2}
    for name, mode, q, out, lse, n_q, fill in (
            ("draft", qs.QS_DRAFT_UPPER4, r.qd[0], r.od[0], None, 1, r.f1 + 1),
            ("verify", qs.QS_VERIFY_INT8, r.qv, r.ov, r.lse, GAMMA + 1, r.f1 + GAMMA + 1)):
        us = time_calls(torch, lambda: qs.qs_attn_decode(r.cache, mode, q, r.scale, out, lse, r.ws),
                        lambda: r.set_state(r.ng1, fill), it, l2)
        nb = sum(attn_bytes(int(n), int(f), n_q, mode == qs.QS_DRAFT_UPPER4, w.H, 1, 2)
                 for n, f in zip(r.ng1, fill))
        res[name + "_us"] = round(us, 2)
        res[name + "_gbs"] = round(nb / us / 1e3, 1)
    assert np.all(qs.qs_get_errors(r.cache) == 0)
    del r
    return res


def gqa_calls(torch, qs, synthetic, l2, it):
    """Grouped-query decode attention on the Llama-3.1-8B shape (8 KV heads,
    32 query heads, 32k context): per-call draft (4 rows per KV head) and
    5-query verify (20 rows) times and GB/s, L2 evicted before each call."""
    w = synthetic.llama31_8b_32k()
    T = w.context[0]
    k, v = synthetic.kv_tokens(w, 0, 0, T)
    cache = qs.Cache(1, w.H, w.n_groups[0] + 1)
    qs.qs_prefill(cache, torch.from_numpy(k[None]).cuda(), torch.from_numpy(v[None]).cuda(),
                  torch.tensor([T], dtype=torch.int32, device="cuda"))
    res = {"workload": w.name}
    for call, (name, mode, n_q) in enumerate((("draft", qs.QS_DRAFT_UPPER4, 1),
                                              ("verify", qs.QS_VERIFY_INT8, GAMMA + 1))):
        q = torch.from_numpy(synthetic.queries(w, call, n_q)).cuda()
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
        ws = torch.empty(qs.qs_attn_workspace_size_gqa(cache, n_q, w.group), dtype=torch.uint8,
                         device="cuda")
        us = time_calls(torch, lambda: qs.qs_attn_decode_gqa(cache, mode, q, w.group, 1 / np.sqrt(w.D),
                                                              out, lse, ws), lambda: None, it, l2)
        nb = attn_bytes(w.n_groups[0], w.fill[0], n_q, mode == qs.QS_DRAFT_UPPER4, w.H, w.group)
        res[name + "_us"] = round(us, 2)
        res[name + "_gbs"] = round(nb / us / 1e3, 1)
    assert np.all(qs.qs_get_errors(cache) == 0)
    del cache
    return res


def native(args):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    from hierarchical_quantized_kv_gb300 import qs, synthetic
    w = synthetic.CONFIGS[args.config](seed=rank)
    r = Round(torch, w, seed=rank)
    peak, peak_kind = load_peaks()

    for s in range(args.warmup):
        r.step(s)
    torch.cuda.synchronize()
    # one CUDA graph per distinct step (the seeded accepted counts cycle with
    # period len(r.drops)); each replay launches the step's kernels
    graphs = [capture(torch, lambda s=s: r.step(s)) for s in range(len(r.drops))]
    for s in range(args.warmup):
        graphs[s % len(graphs)].replay()
    torch.cuda.synchronize()

    reader = nvml_reader(torch, local)
    sampler = ClockSampler(reader=reader) if reader is not None else ClockSampler(smi_index=local)
    time.sleep(0.3 if reader is None else 0.02)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    torch.cuda.nvtx.range_push("timed_steps")  # lets a profiler select the timed launches
    ev0.record()
    for s in range(args.steps):
        graphs[s % len(graphs)].replay()
    ev1.record()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        dist.barrier()
    ms = rank_max(dist, world, ev0.elapsed_time(ev1) / args.steps, "cuda")
    note = "inside timed region"
    t_end = t1
    if sampler.count(t0, t1) < 2:
        # a region shorter than two sampling periods: the same step loop runs
        # on (untimed) until two samples have been taken since it started
        note = ("timed region (%.1f ms) shorter than two sampling periods; samples from its start "
                "through the same graph replays continued right after it" % ((t1 - t0) * 1e3))
        deadline = time.time() + 2.0
        s = args.steps
        while sampler.count(t0, time.time()) < 2 and time.time() < deadline:
            for _ in range(20):
                graphs[s % len(graphs)].replay()
                s += 1
            torch.cuda.synchronize()
        t_end = time.time()
    sampler.stop()
    clocks = sampler.summary(t0, t_end, note)

    # per-call timing with L2 flushed (draft, verify, flush)
    l2 = torch.ones(64 << 20, dtype=torch.float32, device="cuda")  # 256 MB
    it = args.call_iters
    draft_us = time_calls(torch, lambda: qs.qs_attn_decode(r.cache, qs.QS_DRAFT_UPPER4, r.qd[0], r.scale,
                                                           r.od[0], None, r.ws),
                          lambda: r.set_state(r.ng1, r.f1 + 1), it, l2)
    verify_us = time_calls(torch, lambda: qs.qs_attn_decode(r.cache, qs.QS_VERIFY_INT8, r.qv, r.scale,
                                                            r.ov, r.lse, r.ws),
                           lambda: r.set_state(r.ng1, r.f1 + GAMMA + 1), it, l2)
    flush_us = time_calls(torch, lambda: qs.qs_quantize_flush(r.cache, None),
                          lambda: r.cache.state.copy_(r.state0), it, l2)
    r.cache.state.copy_(r.state0)
    # bulk prefill of the whole prompt (one sequence of the workload) into a
    # second cache: one call quantizes every group and fills the buffer
    prefill_us = prefill_gbs = None
    if w.B == 1:
        T = w.context[0]
        kp, vp = synthetic.kv_tokens(w, 0, 0, T)
        kp = torch.from_numpy(kp[None]).cuda()
        vp = torch.from_numpy(vp[None]).cuda()
        lens = torch.tensor([T], dtype=torch.int32, device="cuda")
        pc = qs.Cache(1, w.H, r.cache.cap)
        prefill_us = time_calls(torch, lambda: qs.qs_prefill(pc, kp, vp, lens),
                                lambda: qs.qs_state_reset(pc), it, l2)
        st_p = pc.state[0, :2].cpu().numpy()
        ng_p = -(-(T - 2 * w.G) // w.G) if T > 2 * w.G else 0
        assert st_p[0] == ng_p and st_p[1] == T - ng_p * w.G, st_p
        prefill_gbs = prefill_bytes(T, w.H) / prefill_us / 1e3
        del kp, vp, pc
    main_32k = w.name == synthetic.llama_32k().name
    gqa = gqa_calls(torch, qs, synthetic, l2, it) if main_32k else None
    two_bit = two_bit_calls(torch, qs, synthetic, w, l2, it) if main_32k else None
    # speculative acceptance for the round (synthetic probabilities over a
    # 32,000-token vocabulary): accept/reject, the emitted token, n_drop
    V = 32000
    g_ = torch.Generator(device="cuda").manual_seed(0)
    pp = torch.softmax(torch.randn((w.B, GAMMA + 1, V), device="cuda", generator=g_), dim=-1)
    qq = torch.softmax(torch.randn((w.B, GAMMA, V), device="cuda", generator=g_), dim=-1)
    dr = torch.randint(0, V, (w.B, GAMMA), device="cuda", dtype=torch.int32, generator=g_)
    uu = torch.rand((w.B, GAMMA), device="cuda", generator=g_)
    ee = torch.empty((w.B, V), device="cuda").exponential_(generator=g_)
    sa = [torch.empty(w.B, dtype=torch.int32, device="cuda") for _ in range(3)]
    spec_us = time_calls(torch, lambda: qs.qs_spec_accept(pp, qq, dr, uu, ee, *sa), lambda: None, it,
                         l2)
    del l2
    draft_b, verify_b = r.bytes["draft"][0], r.bytes["verify"]
    draft_gbs, verify_gbs = draft_b / draft_us / 1e3, verify_b / verify_us / 1e3
    # The roofline's launch durations: the attention calls inside the step
    launch, launch_how = in_step_launch_times(torch, r, max(12, min(args.steps, 60)))
    draft_launch_us = float(np.mean(launch["draft_seq"]))
    draft_call_us = float(np.mean(launch["draft"]))
    verify_launch_us = float(np.mean(launch["verify"]))
    draft_marg_us = verify_marg_us = None
    if r.fused:
        draft_marg_us = marginal_us(torch, r, "draft", graphs, max(100, args.steps))
        verify_marg_us = marginal_us(torch, r, "verify", graphs, max(100, args.steps))
    draft_b_mean = float(np.mean(r.bytes["draft"]))
    # dominant kernel by device time within a step
    dominant = ("draft", draft_b_mean / draft_launch_us / 1e3, draft_launch_us) \
        if GAMMA * draft_launch_us >= verify_launch_us else \
        ("verify", verify_b / verify_launch_us / 1e3, verify_launch_us)

    # end to end through host buffers: each step copies its inputs from pinned
    # host memory, runs, copies its outputs back, and the host waits for them.
    # e2e: the step's calls made through the C ABI from Python every step (no
    # graph); e2e_graph: the same step replayed from a CUDA graph.
    host = HostIO(torch, r)
    e_steps = max(1, min(args.steps, 500))
    for s in range(3):
        r.step(s, host)
        torch.cuda.current_stream().synchronize()
    te0 = time.perf_counter()
    for s in range(e_steps):
        r.step(s, host)
        torch.cuda.current_stream().synchronize()  # the host reads the step's result
    e2e_ms = rank_max(dist, world, (time.perf_counter() - te0) * 1e3 / e_steps, "cuda")
    egraphs = [capture(torch, lambda s=s: r.step(s, host)) for s in range(len(r.drops))]
    for s in range(3):
        egraphs[s % len(egraphs)].replay()
        torch.cuda.current_stream().synchronize()
    te0 = time.perf_counter()
    for s in range(e_steps):
        egraphs[s % len(egraphs)].replay()
        torch.cuda.current_stream().synchronize()
    e2e_graph_ms = rank_max(dist, world, (time.perf_counter() - te0) * 1e3 / e_steps, "cuda")
    del egraphs, graphs

    errs = qs.qs_get_errors(r.cache)
    assert np.all(errs == 0), errs
    step_bytes, flushing = r.step_bytes, int(r.plan["mask"].sum())
    launches = r.launches_per_step
    ng_att = int(np.max(r.ng1))
    del r
    torch.cuda.empty_cache()
    configs = {}
    if not args.no_configs and rank == 0 and world == 1:
        for name in ("tiny", "128k", "batched32k", "ragged"):
            if name != args.config:
                configs[name] = config_round(torch, qs, synthetic, name, peak)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, budget_s=args.cpu_budget)
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return
    gbs = aggregate_gbs(step_bytes, world, ms)
    line = {
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "us_per_step": round(ms * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16xf16->f32 (u4 / u8 codes)", "data": "synthetic",
        "config": {"workload": w.name + " speculative round (gamma=4: flush, 4x(append 1 + draft 1q), "
                               "rollback 4, append 5, verify 5q, rollback 4-a)",
                   "B": w.B, "H": w.H, "D": w.D, "G": w.G, "context": w.context[0],
                   "quantized_groups_at_attention": ng_att,
                   "bytes_per_step": step_bytes, "flushing_sequences": flushing,
                   "l2": "step: inputs larger than L2 (%.0f MB of planes per step); per-call numbers: "
                         "L2 evicted before each call by a 256 MB read" % (step_bytes / 1e6),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "draft_in_step_us": round(draft_launch_us, 2), "verify_in_step_us": round(verify_launch_us, 2),
        "draft_in_step_events_per_call_us": round(draft_call_us, 2),
        "draft_marginal_us": None if draft_marg_us is None else round(draft_marg_us, 2),
        "verify_marginal_us": None if verify_marg_us is None else round(verify_marg_us, 2),
        "draft_us": round(draft_us, 2), "draft_gbs": round(draft_gbs, 1),
        "verify_us": round(verify_us, 2), "verify_gbs": round(verify_gbs, 1),
        "flush_us": round(flush_us, 2),
        "prefill_us": None if prefill_us is None else round(prefill_us, 2),
        "prefill_gbs": None if prefill_gbs is None else round(prefill_gbs, 1),
        "spec_accept_us": round(spec_us, 2),
        "gqa": gqa,
        "two_bit_draft": two_bit,
        "roofline": {"bound": "hbm", "kernel": "qs_attn_decode %s (split_kernel: split-KV attention + LSE merge, one launch)" % dominant[0],
                     "launch_us": round(dominant[2], 2),
                     "launch_timing": launch_how + (
                         "; events around the step's run of %d consecutive draft launches, per "
                         "launch (mean of %d runs); events around each single call instead: %.2f us"
                         % (GAMMA, len(launch["draft_seq"]), draft_call_us)
                         if dominant[0] == "draft" else
                         " (mean of %d calls)" % len(launch["verify"])),
                     "achieved": round(dominant[1], 1), "peak": peak,
                     "peak_kind": "%s hbm_gbs (copy, burst)" % peak_kind, "unit": "GB/s",
                     "frac": round(dominant[1] / peak, 4), "traffic": stored_traffic(dominant[0]),
                     "marginal_us": None if draft_marg_us is None else
                     round(draft_marg_us if dominant[0] == "draft" else verify_marg_us, 2),
                     "marginal_frac": None if draft_marg_us is None else
                     round((draft_b_mean if dominant[0] == "draft" else verify_b)
                           / (draft_marg_us if dominant[0] == "draft" else verify_marg_us)
                           / 1e3 / peak, 4),
                     "marginal_timing": "the step's graphs against the same step with one more "
                                        "such call after each, graph-replayed; difference per "
                                        "added call (overlap of consecutive launches included)"},
        "e2e": {"value": round(aggregate_gbs(step_bytes, world, e2e_ms), 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": host.h2d_bytes,
                "d2h_bytes_per_step": host.d2h_bytes,
                "how": "every step: one pinned H2D copy of the step's inputs, the step's %d calls "
                       "through the C ABI (ctypes, no graph), one D2H copy of its outputs, a host "
                       "wait" % launches},
        "e2e_graph": {"value": round(aggregate_gbs(step_bytes, world, e2e_graph_ms), 1),
                      "unit": "GB/s", "ms_per_step": round(e2e_graph_ms, 4),
                      "how": "the same step, copies included, replayed from a CUDA graph"},
        "configs": configs,
        "gpu_launches": launches * args.steps,
        "launch": "CUDA graph replay of each step (one graph per distinct step); the flush "
                  "decides its own mask and each attention call appends its tokens in the same "
                  "launch (qs_quantize_flush_due, qs_attn_decode_append)",
        "clocks": clocks,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------- CPU oracle arm

def cpu_sample(w, heads):
    """Oracle state for a sample of heads of sequence 0 at the step's start."""
    import oracle
    from hierarchical_quantized_kv_gb300 import synthetic
    oc = oracle.OracleCache(1, len(heads), w.D, w.G, w.n_groups[0] + 2)

    def tokens(b, t0, n):
        k, v = synthetic.kv_tokens(w, 0, t0, n)
        return k[heads], v[heads]

    oracle.prefill(oc, tokens, [w.n_groups[0]], [w.fill[0]])
    return oc


def cpu_step(oc, w, s, rng):
    """The benchmark step's work on the oracle (all of it, on the sampled heads).
    Like the device step, it ends by restoring the counters alone, so every
    step flushes into the same group slot and attends over the same lengths."""
    from hierarchical_quantized_kv_gb300 import synthetic
    H, D = oc.H, w.D
    saved = oc.state.copy()
    oc.flush(oc.need_flush(GAMMA + 1))
    for i in range(GAMMA):
        k = rng.standard_normal((1, H, 1, D)).astype(np.float16)
        oc.append(k, k)
        oc.attn(rng.standard_normal((1, H, 1, D)).astype(np.float16), upper_only=True)
    oc.rollback([GAMMA])
    k = rng.standard_normal((1, H, GAMMA + 1, D)).astype(np.float16)
    oc.append(k, k)
    oc.attn(rng.standard_normal((1, H, GAMMA + 1, D)).astype(np.float16), upper_only=False)
    oc.rollback([GAMMA - int(synthetic.accepted_counts(w, s)[0])])
    oc.state[:] = saved


def sample_heads(w):
    """Heads of sequence 0 the oracle sample covers: one per oracle thread (its
    attention runs one (sequence, head) per thread), at most all of them."""
    import oracle
    return list(range(min(w.H, oracle.num_threads())))


def sample_step_bytes(w, n_heads):
    """Algorithmic bytes of one step on the oracle sample: sequence 0's
    counters, n_heads of its heads (the flush counted only if it is due)."""
    return round_plan([w.n_groups[0]], [w.fill[0]], n_heads)["step"]


def cpu_baseline(w, budget_s=15.0):
    heads = sample_heads(w)
    oc = cpu_sample(w, heads)
    rng = np.random.default_rng(5)
    BH = len(heads)
    step_bytes = sample_step_bytes(w, BH)
    n, t0 = 0, time.perf_counter()
    while True:
        cpu_step(oc, w, n, rng)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 20:
            break
    return {"value": round(step_bytes * n / el / 1e9, 4), "unit": "GB/s", "cores": BH,
            "kind": "oracle",
            "sample": "%d benchmark steps on %d of %d heads (sequence 0), %.1f s; fp64 attention "
                      "on %d threads (one head each), the rest of the step on one"
                      % (n, BH, w.H, el, BH),
            "s_per_step_sample": round(el / n, 4)}


def reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from hierarchical_quantized_kv_gb300 import synthetic
    oracle.build.build()
    w = synthetic.CONFIGS[args.config]()
    heads = sample_heads(w)
    oc = cpu_sample(w, heads)
    rng = np.random.default_rng(5)
    BH = len(heads)
    step_bytes = sample_step_bytes(w, BH)
    for s in range(args.warmup):
        cpu_step(oc, w, s, rng)
    t0 = time.perf_counter()
    for s in range(args.steps):
        cpu_step(oc, w, s, rng)
    el = time.perf_counter() - t0
    ms = el * 1e3 / args.steps
    val = round(step_bytes / (ms * 1e-3) / 1e9, 4)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name + " speculative round (gamma=4), bounded CPU sample",
                       "B": w.B, "H": w.H, "D": w.D, "G": w.G, "context": w.context[0],
                       "sample_heads": BH},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": BH,
                             "kind": "oracle",
                             "sample": "each step: the full step's work on %d of %d heads; fp64 "
                                       "attention on %d threads (one head each), the rest on one"
                                       % (BH, w.H, BH)},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def profile(args):
    """A short run for ncu: set up the workload, then ``--profile-calls``
    calls of one kind (draft | verify | flush | step) and nothing else."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from hierarchical_quantized_kv_gb300 import qs, synthetic
    if args.profile.startswith("gqa_"):
        return profile_gqa(args, torch, qs, synthetic)
    w = synthetic.CONFIGS[args.config]()
    r = Round(torch, w, seed=0)
    for i in range(args.warmup if args.profile == "step" else 0):
        r.step(i)
    if args.profile == "prefill":
        T = w.context[0]
        kp, vp = synthetic.kv_tokens(w, 0, 0, T)
        kp, vp = torch.from_numpy(kp[None]).cuda(), torch.from_numpy(vp[None]).cuda()
        lens = torch.tensor([T], dtype=torch.int32, device="cuda")
        pc = qs.Cache(1, w.H, r.cache.cap)
    for i in range(args.profile_calls):
        if args.profile == "draft":
            r.set_state(r.ng1, r.f1 + 1)
            qs.qs_attn_decode(r.cache, qs.QS_DRAFT_UPPER4, r.qd[0], r.scale, r.od[0], None, r.ws)
        elif args.profile == "verify":
            r.set_state(r.ng1, r.f1 + GAMMA + 1)
            qs.qs_attn_decode(r.cache, qs.QS_VERIFY_INT8, r.qv, r.scale, r.ov, r.lse, r.ws)
        elif args.profile == "flush":
            r.cache.state.copy_(r.state0)
            qs.qs_quantize_flush(r.cache, None)
        elif args.profile == "prefill":
            qs.qs_state_reset(pc)
            qs.qs_prefill(pc, kp, vp, lens)
        else:
            r.step(i)
    torch.cuda.synchronize()
    assert np.all(qs.qs_get_errors(r.cache) == 0)
    print("profile run ok: %d %s calls on %s" % (args.profile_calls, args.profile, w.name))


def profile_gqa(args, torch, qs, synthetic):
    """--profile gqa_draft | gqa_verify: the Llama-3.1-8B 32k shape (8 KV heads,
    32 query heads), one prefill, then the calls."""
    w = synthetic.llama31_8b_32k()
    T = w.context[0]
    k, v = synthetic.kv_tokens(w, 0, 0, T)
    cache = qs.Cache(1, w.H, w.n_groups[0] + 1)
    qs.qs_prefill(cache, torch.from_numpy(k[None]).cuda(), torch.from_numpy(v[None]).cuda(),
                  torch.tensor([T], dtype=torch.int32, device="cuda"))
    draft = args.profile == "gqa_draft"
    n_q = 1 if draft else GAMMA + 1
    mode = qs.QS_DRAFT_UPPER4 if draft else qs.QS_VERIFY_INT8
    q = torch.from_numpy(synthetic.queries(w, 0, n_q)).cuda()
    out = torch.empty_like(q)
    ws = torch.empty(qs.qs_attn_workspace_size_gqa(cache, n_q, w.group), dtype=torch.uint8,
                     device="cuda")
    for _ in range(args.profile_calls):
        qs.qs_attn_decode_gqa(cache, mode, q, w.group, 1 / np.sqrt(w.D), out, None, ws)
    torch.cuda.synchronize()
    assert np.all(qs.qs_get_errors(cache) == 0)
    print("profile run ok: %d %s calls on %s" % (args.profile_calls, args.profile, w.name))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="32k")
    ap.add_argument("--call-iters", type=int, default=30)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the rounds on the other workloads")
    ap.add_argument("--profile", choices=["draft", "verify", "flush", "prefill", "step", "gqa_draft",
                                          "gqa_verify"])
    ap.add_argument("--profile-calls", type=int, default=3)
    args = ap.parse_args()
    if args.profile:
        profile(args)
    elif args.impl == "reference":
        if args.steps > 20:  # each oracle step is a bounded CPU sample (about a second)
            args.steps = 20
        args.warmup = min(args.warmup, 3)
        reference(args)
    else:
        native(args)


if __name__ == "__main__":
    main()
