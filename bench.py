"""Benchmark: GLANCE verify rounds per second on one GB300 (or N replicas).

One step = one verify round over the full36 workload (Qwen3-VL-8B geometry):
draft-to-tree (L = 15 offsets over V = 151936, N = 63), ancestor-masked tree
attention in all 36 layers against a T = 4096 prefix, LM head [64, 4096] x
[4096, 151936] with fused argmax / top-2 gap, acceptance walk and KV commit
over the 36 layers. Inputs are seeded synthetic data resident in HBM; each
step streams ~1.9 GB of distinct data (more than the 129 MB L2), so no L2
flush is inserted. The round is captured in a CUDA graph and replayed.

Prints one JSON line (see the keys below). `--impl reference` times the CPU
oracle on a bounded sample of the same workload instead.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "verify rounds/s at N=63 (tree+attn+LMhead+walk); HBM GB/s & TC util vs peak"
FULL36 = dict(name="full36", T=4096, N=63, L=15, V=151936, d=4096, n_layers=36, Hq=32, Hkv=8,
              D=128, path_depth=(3, 15))
SMALL = dict(name="small", T=512, N=31, L=15, V=16384, d=512, n_layers=4, Hq=32, Hkv=8, D=128,
             path_depth=(3, 15))
FORWARD36 = dict(name="forward36", T=4096, N=63, L=15, V=151936, d=4096, n_layers=36, Hq=32, Hkv=8,
                 D=128, inter=12288, rope_theta=1e6, eps=1e-6, path_depth=(3, 15))
ENTROPY36 = dict(name="entropy36", T=2048, L=15, V=151936, d=4096, n_layers=36, Hq=32, Hkv=8, D=128,
                 entropy=(0.3, 1.5, 4.0), N_set=(31, 63, 127, 255))
VERIFY1 = dict(name="verify1", T=1024, N=31, L=15, V=151936, n_layers=1, Hq=32, Hkv=8, D=128)
RAGGED8 = dict(name="ragged8", B=8, T_range=(512, 8192), entropy=(0.3, 1.5, 4.0), N=63, L=15,
               V=151936, d=4096, n_layers=36, Hq=32, Hkv=8, D=128, path_depth=(3, 15))


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sust=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, src="fallback")


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# one ncu capture of the full36 workload. A figure holds only for the kernel
# sources it was taken on: `digest` is the first 16 hex digits of the sha256 of
# the listed files, and a changed source reports traffic null.
CSRC = os.path.join("tree_verified_block_gb300", "csrc")
NCU_TRAFFIC = {
    "glance_tree_attention": dict(bytes=17_901_312, digest="0a37add0e235cce0",
                                  files=["tree_attention.cu", "glance_internal.cuh"],
                                  profile="profiles/tree_attention_full36.md"),
    "glance_lmhead_argmax": dict(bytes=1_246_313_472 + 3_105_536, digest="21b18a1285869c18",
                                 files=["lmhead.cu", "glance_internal.cuh"],
                                 profile="profiles/lmhead_argmax_full36.md"),
}


def source_digest(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel):
    e = NCU_TRAFFIC.get(kernel)
    if e is None or source_digest(e["files"]) != e["digest"]:
        return None
    return e["bytes"]


def workload_config(cfg):
    return {"workload": f"{cfg['name']}: Qwen3-VL-8B verify round, T={cfg['T']}, N={cfg['N']}, "
                        f"L={cfg['L']}, V={cfg['V']}, d={cfg['d']}, {cfg['n_layers']} layers, "
                        f"{cfg['Hq']}/{cfg['Hkv']} heads x {cfg['D']}",
            "T": cfg["T"], "N": cfg["N"], "L": cfg["L"], "V": cfg["V"], "d": cfg["d"],
            "n_layers": cfg["n_layers"], "parallelism": "one GPU (the path is per request; more GPUs would run replicas)",
            "l2": "no flush: each step streams ~1.9 GB of distinct inputs (> 129 MB L2)",
            "cuda_graph": True}


# ------------------------------------------------------------------ workload

class Workload:
    """Device-resident inputs of one verify round plus their host copies."""

    def __init__(self, cfg, dev, seed=3000, keep_host=True):
        import torch
        import tree_verified_block_gb300 as g
        self.cfg, self.dev, self.g = cfg, dev, g
        c = cfg
        R = c["N"] + 1
        self.R = R
        self.t_cap = c["T"] + R + 64
        gen = W.rng(seed)
        self.x = W.draft_logits_planted(c["L"], c["V"], seed=seed + 1)
        self.q_bits = [W.normal_bf16(gen, (R, c["Hq"], c["D"])) for _ in range(c["n_layers"])]
        self.k_bits, self.v_bits = [], []
        for _ in range(c["n_layers"]):
            self.k_bits.append(W.normal_bf16(gen, (c["Hkv"], self.t_cap, c["D"])))
            self.v_bits.append(W.normal_bf16(gen, (c["Hkv"], self.t_cap, c["D"])))
        self.W_bits = W.normal_bf16(gen, (c["d"], c["V"]), std=0.02)
        bf = lambda b: torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16)
        self.x_dev = torch.from_numpy(self.x).to(dev)
        self.q = [bf(b) for b in self.q_bits]
        self.k = [bf(b) for b in self.k_bits]
        self.v = [bf(b) for b in self.v_bits]
        self.W = bf(self.W_bits)
        # W packed once as the LM head's stage images (a model constant, like
        # the weights themselves); the round reads it through the packed call
        self.Wp = torch.empty(g.lmhead_packed_w_bytes(c["d"], c["V"]), dtype=torch.uint8, device=dev)
        g.lmhead_pack_w(self.W, self.Wp)
        self.t0 = torch.tensor([c["T"]], dtype=torch.int32, device=dev)
        self.t_len = self.t0.clone()
        self.root = torch.tensor([int(gen.integers(0, c["V"]))], dtype=torch.int32, device=dev)
        self.layers = [g.KVLayer(k, v, self.t_len) for k, v in zip(self.k, self.v)]
        self.tree = g.Tree(c["N"], c["L"], dev)
        self.out = [torch.empty_like(q) for q in self.q]
        self.argmax = torch.empty(R, dtype=torch.int32, device=dev)
        self.gap = torch.empty(R, dtype=torch.float32, device=dev)
        self.maxlogit = torch.empty(R, dtype=torch.float32, device=dev)
        self.n_acc = torch.zeros(1, dtype=torch.int32, device=dev)
        self.acc_tok = torch.zeros(c["L"], dtype=torch.int32, device=dev)
        self.new_root = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws_tree = g.workspace(g.build_tree_workspace_bytes(c["L"], c["V"], c["N"]), dev)
        self.ws_attn = g.workspace(g.tree_attention_workspace_bytes(R, c["Hq"], self.layers[0]), dev)
        self.ws_lm = g.workspace(g.lmhead_argmax_workspace_bytes(R, c["d"], c["V"], torch.bfloat16), dev)
        self.ws_c = g.workspace(g.accept_commit_workspace_bytes(c["n_layers"]), dev)
        # h: planted so that the greedy path follows the tree's best child chain
        g.build_tree(self.x_dev, c["N"], self.root, self.t_len, self.tree, self.ws_tree)
        th = self.tree.to_host()
        self.path_rows, self.path_tokens = self._chain(th, gen)
        h = gen.standard_normal((R, c["d"]), dtype=np.float32)
        Wf_cols = lambda toks: W.bf16_bits_to_f32(self.W_bits[:, toks])
        hp = h.copy()
        for r, t in zip(self.path_rows, self.path_tokens):
            col = Wf_cols([t])[:, 0].astype(np.float64)
            hp[r] += (10.0 * col / (col @ col)).astype(np.float32)
        self.h_bits = W.to_bf16_bits(hp)
        self.h = bf(self.h_bits)
        self.tree_host = th
        if not keep_host:
            self.k_bits = self.v_bits = self.W_bits = None

    def _chain(self, th, gen):
        """Rows of the highest-score child chain (depth ~ U{lo..hi}) and the
        greedy tokens that make the walk follow it; the last row gets a token
        that is not one of its children."""
        lo, hi = self.cfg["path_depth"]
        want = int(gen.integers(lo, hi + 1))
        rows, toks = [], []
        u = 0
        for _ in range(want):
            kids = [c for c in range(self.R) if th["parent"][c] == u]
            if not kids:
                break
            c = max(kids, key=lambda k: (th["score"][k], -k))
            rows.append(u)
            toks.append(int(th["token"][c]))
            u = c
        kid_tokens = {int(th["token"][c]) for c in range(self.R) if th["parent"][c] == u}
        t = int(gen.integers(0, self.cfg["V"]))
        while t in kid_tokens:
            t = (t + 1) % self.cfg["V"]
        rows.append(u)
        toks.append(t)
        return rows, toks

    # one verify round, all on the current stream
    def step(self):
        g, c = self.g, self.cfg
        self.t_len.copy_(self.t0)
        g.build_tree(self.x_dev, c["N"], self.root, self.t_len, self.tree, self.ws_tree)
        scale = c["D"] ** -0.5
        for l in range(c["n_layers"]):
            g.tree_attention(self.q[l], self.layers[l], self.tree, scale, self.out[l], self.ws_attn)
        g.lmhead_argmax_packed(self.h, self.Wp, c["V"], self.argmax, self.gap, self.maxlogit, self.ws_lm)
        g.accept_commit(self.tree, self.argmax, self.layers, self.n_acc, self.acc_tok,
                        self.new_root, self.ws_c)

    def launches_per_step(self):
        # one launch per ABI call: build_tree, tree_attention per layer,
        # lmhead_argmax_packed, accept_commit (the t_len reset is a torch copy)
        return 1 + self.cfg["n_layers"] + 1 + 1

    def algorithmic_bytes(self):
        c = self.cfg
        R = self.R
        tree = c["L"] * c["V"] * 4
        attn_layer = (c["T"] + R) * c["Hkv"] * c["D"] * 2 * 2 + 2 * R * c["Hq"] * c["D"] * 2
        lm = c["d"] * c["V"] * 2 + R * c["d"] * 2
        return dict(tree=tree, attn_layer=attn_layer, lmhead=lm)

    def flops(self):
        c = self.cfg
        lm = 2 * self.R * c["d"] * c["V"]
        return dict(lmhead=lm)


class BatchedWorkload:
    """B concurrent requests with ragged prefix lengths T ~ U{512..8192}, each
    with its own draft marginals (entropy 0.3 / 1.5 / 4.0 nats cycled), root,
    N = 63 tree and per-request KV caches; one launch per step over the batch
    and the LM head over the B x 64 stacked rows.

    host=True draws every input with the seeded numpy generators (the oracle
    can recompute from the host copies); host=False draws q, K, V and W with a
    seeded torch generator on the device (same distributions; for timing,
    where 36 layers of ragged caches would take minutes to draw on the host).
    """

    def __init__(self, cfg, dev, seed=5000, host=True, n_layers=None):
        import torch
        import tree_verified_block_gb300 as g
        c = dict(cfg)
        if n_layers is not None:
            c["n_layers"] = n_layers
        self.cfg, self.dev, self.g, self.host = c, dev, g, host
        B, R, D = c["B"], c["N"] + 1, c["D"]
        self.B, self.R = B, R
        gen = W.rng(seed)
        lo, hi = c["T_range"]
        self.T = [int(t) for t in gen.integers(lo, hi + 1, size=B)]
        self.t_cap = [t + R + 64 for t in self.T]
        self.x = np.stack([W.draft_logits_entropy(c["L"], c["V"], c["entropy"][r % len(c["entropy"])],
                                                  seed=seed + 1 + r) for r in range(B)])
        bf = lambda b: torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16)
        if host:
            self.q_bits = [W.normal_bf16(gen, (B, R, c["Hq"], D)) for _ in range(c["n_layers"])]
            self.k_bits = [[W.normal_bf16(gen, (c["Hkv"], self.t_cap[r], D)) for r in range(B)]
                           for _ in range(c["n_layers"])]
            self.v_bits = [[W.normal_bf16(gen, (c["Hkv"], self.t_cap[r], D)) for r in range(B)]
                           for _ in range(c["n_layers"])]
            self.W_bits = W.normal_bf16(gen, (c["d"], c["V"]), std=0.02)
            self.q = [bf(b) for b in self.q_bits]
            self.k = [[bf(b) for b in kl] for kl in self.k_bits]
            self.v = [[bf(b) for b in vl] for vl in self.v_bits]
            self.W = bf(self.W_bits)
            h = gen.standard_normal((B * R, c["d"]), dtype=np.float32)
            self.h_f32 = torch.from_numpy(h).to(dev)
        else:
            tg = torch.Generator(device=dev)
            tg.manual_seed(seed)
            rn = lambda *shape, std=1.0: (torch.randn(*shape, generator=tg, device=dev) * std).to(torch.bfloat16)
            self.q = [rn(B, R, c["Hq"], D) for _ in range(c["n_layers"])]
            self.k = [[rn(c["Hkv"], self.t_cap[r], D) for r in range(B)] for _ in range(c["n_layers"])]
            self.v = [[rn(c["Hkv"], self.t_cap[r], D) for r in range(B)] for _ in range(c["n_layers"])]
            self.W = rn(c["d"], c["V"], std=0.02)
            self.h_f32 = torch.randn(B * R, c["d"], generator=tg, device=dev)
            self.q_bits = self.k_bits = self.v_bits = self.W_bits = None
        self.x_dev = torch.from_numpy(self.x.astype(np.float32)).to(dev)
        self.t0 = torch.tensor(self.T, dtype=torch.int32, device=dev)
        self.t_len = self.t0.clone()
        self.root = torch.from_numpy(gen.integers(0, c["V"], size=B).astype(np.int32)).to(dev)
        # layers[l][r] for attention, by_req[r][l] for the commit
        self.layers = [[g.KVLayer(self.k[l][r], self.v[l][r], self.t_len[r:r + 1]) for r in range(B)]
                       for l in range(c["n_layers"])]
        self.by_req = [[self.layers[l][r] for l in range(c["n_layers"])] for r in range(B)]
        self.trees = [g.Tree(c["N"], c["L"], dev) for _ in range(B)]
        self.out = [torch.empty_like(q) for q in self.q]
        M = B * R
        self.argmax = torch.empty(M, dtype=torch.int32, device=dev)
        self.gap = torch.empty(M, dtype=torch.float32, device=dev)
        self.maxlogit = torch.empty(M, dtype=torch.float32, device=dev)
        self.n_acc = torch.zeros(B, dtype=torch.int32, device=dev)
        self.acc_tok = torch.zeros((B, c["L"]), dtype=torch.int32, device=dev)
        self.new_root = torch.zeros(B, dtype=torch.int32, device=dev)
        self.ws_tree = g.workspace(g.build_tree_batched_workspace_bytes(B, c["L"], c["V"], c["N"]), dev)
        self.ws_attn = g.workspace(g.tree_attention_batched_workspace_bytes(R, c["Hq"], self.layers[0]), dev)
        self.ws_lm = g.workspace(g.lmhead_argmax_workspace_bytes(M, c["d"], c["V"], torch.bfloat16), dev)
        self.ws_c = g.workspace(g.accept_commit_batched_workspace_bytes(B, c["n_layers"]), dev)
        # h: each request's rows planted so that its walk follows its best chain
        g.build_tree_batched(self.x_dev, c["N"], self.root, self.t_len, self.trees, self.ws_tree)
        self.tree_host = [t.to_host() for t in self.trees]
        self.path_rows, self.path_tokens = [], []
        hp = self.h_f32.clone()
        for r in range(B):
            rows, toks = Workload._chain(self, self.tree_host[r], gen)
            self.path_rows.append(rows)
            self.path_tokens.append(toks)
            for u, t in zip(rows, toks):
                col = self.W[:, t].double()
                hp[r * R + u] += (10.0 * col / (col @ col)).float()
        self.h = hp.to(torch.bfloat16)
        self.h_bits = self.h.view(torch.int16).cpu().numpy().view(np.uint16) if host else None

    def step(self):
        g, c = self.g, self.cfg
        self.t_len.copy_(self.t0)
        g.build_tree_batched(self.x_dev, c["N"], self.root, self.t_len, self.trees, self.ws_tree)
        scale = c["D"] ** -0.5
        for l in range(c["n_layers"]):
            g.tree_attention_batched(self.q[l], self.layers[l], self.trees, scale, self.out[l],
                                     self.ws_attn)
        g.lmhead_argmax(self.h, self.W, self.argmax, self.gap, self.maxlogit, self.ws_lm)
        g.accept_commit_batched(self.trees, self.argmax, self.by_req, self.n_acc, self.acc_tok,
                                self.new_root, self.ws_c)

    def algorithmic_bytes(self):
        c = self.cfg
        R = self.R
        attn = sum((t + R) * c["Hkv"] * c["D"] * 2 * 2 for t in self.T) + 2 * self.B * R * c["Hq"] * c["D"] * 2
        return dict(tree=self.B * c["L"] * c["V"] * 4, attn_layer=attn,
                    lmhead=c["d"] * c["V"] * 2 + self.B * R * c["d"] * 2)

    def flops(self):
        c = self.cfg
        return dict(lmhead=2 * self.B * self.R * c["d"] * c["V"])


# ------------------------------------------------------------------ clocks

class _NvmlClocks:
    """SM clock and clock-event reasons read through NVML (libnvidia-ml, read-only
    queries), for the device torch calls `dev`; matched by PCI bus id."""
    # NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*)
    BITS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
            0x4: "sw_power_cap"}

    def __init__(self, dev):
        import ctypes
        import torch
        self.c = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        pr = torch.cuda.get_device_properties(dev)
        bus = getattr(pr, "pci_bus_id", None)
        ok = -1
        if bus is not None:
            bid = f"{getattr(pr, 'pci_domain_id', 0):08x}:{bus:02x}:{getattr(pr, 'pci_device_id', 0):02x}.0"
            ok = lib.nvmlDeviceGetHandleByPciBusId_v2(bid.encode(), ctypes.byref(self.h))
        if ok != 0:
            ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(dev.index or 0), ctypes.byref(self.h))
        if ok != 0:
            raise RuntimeError("no NVML handle")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.max_mhz = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0 else None

    def sample(self):
        c = self.c
        mhz, rs = c.c_uint(), c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, c.byref(mhz)) != 0:
            return None
        if self.reasons_fn(self.h, c.byref(rs)) != 0:
            rs.value = 0
        return float(mhz.value), [n for b, n in self.BITS.items() if rs.value & b]


class ClockSampler:
    """SM clocks and throttle reasons sampled during the timed region: NVML
    every 5 ms from a host thread, else `nvidia-smi -lms 200`."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, dev):
        self.dev = dev
        self.proc = None
        self.nvml = None
        self.lines = []
        self.samples = []
        self.stop = threading.Event()

    def __enter__(self):
        try:
            self.nvml = _NvmlClocks(self.dev)
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev.index or 0), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _poll(self):
        while not self.stop.is_set():
            s = self.nvml.sample()
            if s is not None:
                self.samples.append(s)
            time.sleep(0.005)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        self.stop.set()
        if self.nvml is not None:
            self.thread.join(timeout=2)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        if self.nvml is not None:
            for mhz, rs in self.samples:
                sm.append(mhz)
                reasons.update(rs)
            mx = self.nvml.max_mhz
            src = "nvml 5 ms"
        else:
            for ln in self.lines:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(self.NAMES, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
            src = "nvidia-smi 200 ms"
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "sampler": src}


class ForwardWorkload:
    """The whole verify forward of one round on a Qwen3-8B-shaped target:
    tree build, then per layer the dense calls around tree attention (QKV with
    q/k norm and RoPE into the layer's cache, attention, output projection,
    SwiGLU, down projection; RMSNorm row scales from the residual projections'
    row sums of squares), the LM head with argmax on the last layer's rows, and
    the walk + commit. Weights, input rows and K/V are drawn on the device from
    a seeded torch generator (N(0, 0.02) weights, N(0, 1) rows and K/V); the
    RMSNorm gains are taken as already folded into the next projection's rows.
    The final norm's row scale is left out: a positive per-row scale does not
    move a row's argmax."""

    def __init__(self, cfg, dev, seed=7000):
        import torch
        import tree_verified_block_gb300 as g
        self.cfg, self.dev, self.g = cfg, dev, g
        c = cfg
        R = c["N"] + 1
        self.R = R
        t_cap = c["T"] + R + 64
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed)
        bf = dict(dtype=torch.bfloat16, device=dev)

        def w(k, n):
            return (torch.randn(k, n, generator=gen, device=dev) * 0.02).to(torch.bfloat16)

        d, I, D = c["d"], c["inter"], c["D"]
        qkv_cols = (c["Hq"] + 2 * c["Hkv"]) * D
        self.Wqkv = [w(d, qkv_cols) for _ in range(c["n_layers"])]
        self.Wo = [w(c["Hq"] * D, d) for _ in range(c["n_layers"])]
        self.Wg = [w(d, I) for _ in range(c["n_layers"])]
        self.Wu = [w(d, I) for _ in range(c["n_layers"])]
        self.Wd = [w(I, d) for _ in range(c["n_layers"])]
        self.W = w(d, c["V"])
        self.k = [torch.randn(c["Hkv"], t_cap, D, generator=gen, device=dev).to(torch.bfloat16)
                  for _ in range(c["n_layers"])]
        self.v = [torch.randn(c["Hkv"], t_cap, D, generator=gen, device=dev).to(torch.bfloat16)
                  for _ in range(c["n_layers"])]
        self.x_dev = torch.from_numpy(W.draft_logits_planted(c["L"], c["V"], seed=seed + 1)).to(dev)
        self.emb = torch.randn(R, d, generator=gen, device=dev).to(torch.bfloat16)
        self.t0 = torch.tensor([c["T"]], dtype=torch.int32, device=dev)
        self.t_len = self.t0.clone()
        self.root = torch.tensor([1234], dtype=torch.int32, device=dev)
        self.layers = [g.KVLayer(k, v, self.t_len) for k, v in zip(self.k, self.v)]
        self.tree = g.Tree(c["N"], c["L"], dev)
        self.xa = torch.empty(R, d, **bf)
        self.q = torch.empty(R, c["Hq"], D, **bf)
        self.att = torch.empty(R, c["Hq"], D, **bf)
        self.act = torch.empty(R, I, **bf)
        self.ss0 = torch.empty(R, dtype=torch.float32, device=dev)
        self.ss_a = torch.empty(d // 256, R, dtype=torch.float32, device=dev)
        self.ss_b = torch.empty(d // 256, R, dtype=torch.float32, device=dev)
        self.argmax = torch.empty(R, dtype=torch.int32, device=dev)
        self.gap = torch.empty(R, dtype=torch.float32, device=dev)
        self.maxlogit = torch.empty(R, dtype=torch.float32, device=dev)
        self.n_acc = torch.zeros(1, dtype=torch.int32, device=dev)
        self.acc_tok = torch.zeros(c["L"], dtype=torch.int32, device=dev)
        self.new_root = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws_tree = g.workspace(g.build_tree_workspace_bytes(c["L"], c["V"], c["N"]), dev)
        self.ws_attn = g.workspace(g.tree_attention_workspace_bytes(R, c["Hq"], self.layers[0]), dev)
        self.ws_lm = g.workspace(g.lmhead_argmax_workspace_bytes(R, d, c["V"], torch.bfloat16), dev)
        self.ws_c = g.workspace(g.accept_commit_workspace_bytes(c["n_layers"]), dev)

    def layer(self, l):
        """One decoder layer over the packed rows (layer 0 reads the input rows)."""
        g, c = self.g, self.cfg
        x_in, ss_in = (self.emb, self.ss0) if l == 0 else (self.xa, self.ss_b)
        g.dense_qkv(x_in, self.Wqkv[l], c["Hq"], ss_in, None, None, c["eps"], self.tree.pos_id,
                    c["rope_theta"], self.q, self.layers[l])
        g.tree_attention(self.q, self.layers[l], self.tree, c["D"] ** -0.5, self.att, self.ws_attn)
        g.dense_residual(self.att.view(self.R, -1), self.Wo[l], x_in, self.xa, self.ss_a)
        g.dense_swiglu(self.xa, self.Wg[l], self.Wu[l], self.ss_a, c["eps"], self.act)
        g.dense_residual(self.act, self.Wd[l], self.xa, self.xa, self.ss_b)

    def step(self):
        g, c = self.g, self.cfg
        self.t_len.copy_(self.t0)
        g.build_tree(self.x_dev, c["N"], self.root, self.t_len, self.tree, self.ws_tree)
        g.row_sumsq(self.emb, self.ss0)
        for l in range(c["n_layers"]):
            self.layer(l)
        g.lmhead_argmax(self.xa, self.W, self.argmax, self.gap, self.maxlogit, self.ws_lm)
        g.accept_commit(self.tree, self.argmax, self.layers, self.n_acc, self.acc_tok,
                        self.new_root, self.ws_c)

    def launches_per_step(self):
        return 2 + 5 * self.cfg["n_layers"] + 2

    def algorithmic_bytes(self):
        c = self.cfg
        R, d, I, D = self.R, c["d"], c["inter"], c["D"]
        dense = (d * (c["Hq"] + 2 * c["Hkv"]) * D + c["Hq"] * D * d + 3 * d * I) * 2
        attn = (c["T"] + R) * c["Hkv"] * D * 2 * 2 + 2 * R * c["Hq"] * D * 2
        return dict(dense_layer=dense, attn_layer=attn, lmhead=d * c["V"] * 2 + R * d * 2,
                    tree=c["L"] * c["V"] * 4)


# ------------------------------------------------------------------ timing

def graph_time_us(fn, reps=20):
    """Device time of fn's launches, captured in a CUDA graph and replayed
    `reps` times between two events on the launching stream (no host launch
    latency in the measurement)."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    g.replay()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    for _ in range(reps):
        g.replay()
    b.record(s)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / reps


def stage_times(wl, reps=20):
    """Per-stage device times (us), each stage graph-captured and replayed."""
    g, c = wl.g, wl.cfg
    scale = c["D"] ** -0.5
    res = {}

    def tree():
        wl.t_len.copy_(wl.t0)
        g.build_tree(wl.x_dev, c["N"], wl.root, wl.t_len, wl.tree, wl.ws_tree)
    res["tree"] = graph_time_us(tree, reps)
    res["attention_36"] = graph_time_us(
        lambda: [g.tree_attention(wl.q[l], wl.layers[l], wl.tree, scale, wl.out[l], wl.ws_attn)
                 for l in range(c["n_layers"])], reps)
    res["attention_layer"] = graph_time_us(
        lambda: g.tree_attention(wl.q[0], wl.layers[0], wl.tree, scale, wl.out[0], wl.ws_attn), reps * 5)
    res["lmhead"] = graph_time_us(
        lambda: g.lmhead_argmax_packed(wl.h, wl.Wp, c["V"], wl.argmax, wl.gap, wl.maxlogit, wl.ws_lm), reps)

    def commit():
        wl.t_len.copy_(wl.t0)
        g.accept_commit(wl.tree, wl.argmax, wl.layers, wl.n_acc, wl.acc_tok, wl.new_root, wl.ws_c)
    res["commit"] = graph_time_us(commit, reps)
    res["t_reset_copy"] = graph_time_us(lambda: wl.t_len.copy_(wl.t0), reps)
    return res


def run_batched(dev, reps=10):
    """The ragged8 batched round (secondary measurement): whole round and
    per-stage device times from CUDA-graph replays, with each stage's
    fraction of its roof."""
    bw = BatchedWorkload(RAGGED8, dev, seed=5000, host=False)
    g, c = bw.g, bw.cfg
    import torch
    for _ in range(3):
        bw.step()
    torch.cuda.synchronize()
    scale = c["D"] ** -0.5
    st = {"round": graph_time_us(bw.step, reps)}

    def tree():
        bw.t_len.copy_(bw.t0)
        g.build_tree_batched(bw.x_dev, c["N"], bw.root, bw.t_len, bw.trees, bw.ws_tree)
    st["tree"] = graph_time_us(tree, reps)
    st["attention_36"] = graph_time_us(
        lambda: [g.tree_attention_batched(bw.q[l], bw.layers[l], bw.trees, scale, bw.out[l], bw.ws_attn)
                 for l in range(c["n_layers"])], reps)
    st["attention_layer"] = graph_time_us(
        lambda: g.tree_attention_batched(bw.q[0], bw.layers[0], bw.trees, scale, bw.out[0], bw.ws_attn),
        reps * 5)
    st["lmhead_m512"] = graph_time_us(
        lambda: g.lmhead_argmax(bw.h, bw.W, bw.argmax, bw.gap, bw.maxlogit, bw.ws_lm), reps)

    def commit():
        bw.t_len.copy_(bw.t0)
        g.accept_commit_batched(bw.trees, bw.argmax, bw.by_req, bw.n_acc, bw.acc_tok, bw.new_root,
                                bw.ws_c)
    st["commit"] = graph_time_us(commit, reps)
    # the NEXT rows on the same batch: shared-budget trees (half the batch's
    # nodes, entropy-keyed with the pooled law), the LM head with the root
    # entropy and in sampling mode, the gated walk + commit
    M = bw.B * bw.R
    ent = torch.tensor([c["entropy"][r % len(c["entropy"])] for r in range(bw.B)], dtype=torch.float32,
                       device=bw.x_dev.device)
    n_active = torch.zeros(bw.B, dtype=torch.int32, device=bw.x_dev.device)
    ws_sh = g.workspace(g.build_tree_shared_workspace_bytes(bw.B, c["L"], c["V"], c["N"]), bw.x_dev.device)

    def tree_shared():
        bw.t_len.copy_(bw.t0)
        g.build_tree_shared(bw.x_dev, c["N"], bw.B * c["N"] // 2, bw.root, bw.t_len, bw.trees, n_active, ws_sh,
                            root_entropy=ent, law_b0=0.96, law_b1=0.63)
    st["tree_shared"] = graph_time_us(tree_shared, reps)
    entropy = torch.empty(M, dtype=torch.float32, device=bw.x_dev.device)
    st["lmhead_entropy_m512"] = graph_time_us(
        lambda: g.lmhead_argmax_entropy(bw.h, bw.W, bw.argmax, bw.gap, bw.maxlogit, entropy, bw.ws_lm), reps)
    pos = torch.arange(M, dtype=torch.int32, device=bw.x_dev.device)
    seq = torch.zeros(M, dtype=torch.int32, device=bw.x_dev.device)
    drawn = torch.empty(M, dtype=torch.int32, device=bw.x_dev.device)
    st["lmhead_sample_m512"] = graph_time_us(
        lambda: g.lmhead_sample(bw.h, bw.W, 1.0, 1234, pos, seq, drawn, bw.gap, bw.ws_lm), reps)
    gated = torch.zeros(bw.B, dtype=torch.int32, device=bw.x_dev.device)
    g.lmhead_argmax(bw.h, bw.W, bw.argmax, bw.gap, bw.maxlogit, bw.ws_lm)
    tree()  # the full trees again for the walk

    def commit_gated():
        bw.t_len.copy_(bw.t0)
        g.accept_commit_gated_batched(bw.trees, bw.argmax, bw.gap, 1e-3, bw.by_req, bw.n_acc, bw.acc_tok,
                                      bw.new_root, gated, bw.ws_c)
    st["commit_gated"] = graph_time_us(commit_gated, reps)
    pk = peaks()
    by, fl = bw.algorithmic_bytes(), bw.flops()
    lm_tf = fl["lmhead"] / (st["lmhead_m512"] * 1e-6) / 1e12
    out = {"workload": f"ragged8: {c['B']} requests, T in {bw.T}, N={c['N']}, L={c['L']}, "
                       f"V={c['V']}, d={c['d']}, {c['n_layers']} layers, LM head M={bw.B * bw.R}",
           "rounds_per_s": round(1e6 / st["round"], 2),
           "request_rounds_per_s": round(bw.B * 1e6 / st["round"], 2),
           "stages_us": {k: round(v, 2) for k, v in st.items()},
           "attention_layer_hbm_frac": round(by["attn_layer"] * c["n_layers"] / (st["attention_36"] * 1e-6) / 1e9
                                             / pk["hbm"], 4),
           "lmhead_m512_tflops": round(lm_tf, 1),
           "lmhead_m512_tensor_frac": round(lm_tf / pk["bf16"], 4),
           "lmhead_m512_hbm_frac": round(by["lmhead"] / (st["lmhead_m512"] * 1e-6) / 1e9 / pk["hbm"], 4),
           "data": "synthetic, q/K/V/W drawn on the device (seeded torch generator)"}
    return out


def run_forward(dev, reps=10):
    """The whole verify forward (forward36; secondary measurement): the round
    and its stages from CUDA-graph replays, each against the HBM roof of its
    algorithmic bytes."""
    import torch
    fw = ForwardWorkload(FORWARD36, dev)
    c = fw.cfg
    for _ in range(3):
        fw.step()
    torch.cuda.synchronize()
    st = {"round": graph_time_us(fw.step, reps)}
    n = c["n_layers"]
    g = fw.g
    # each stage over all n layers' weights (distinct, > L2 in total), per launch
    per = lambda fn: graph_time_us(lambda: [fn(l) for l in range(n)], reps) / n
    st["layer"] = per(fw.layer)
    st["qkv"] = per(lambda l: g.dense_qkv(fw.xa, fw.Wqkv[l], c["Hq"], fw.ss_b, None, None, c["eps"],
                                          fw.tree.pos_id, c["rope_theta"], fw.q, fw.layers[l]))
    st["attention"] = per(lambda l: g.tree_attention(fw.q, fw.layers[l], fw.tree, c["D"] ** -0.5, fw.att,
                                                     fw.ws_attn))
    st["o_proj"] = per(lambda l: g.dense_residual(fw.att.view(fw.R, -1), fw.Wo[l], fw.emb, fw.xa, fw.ss_a))
    st["swiglu"] = per(lambda l: g.dense_swiglu(fw.xa, fw.Wg[l], fw.Wu[l], fw.ss_a, c["eps"], fw.act))
    st["down_proj"] = per(lambda l: g.dense_residual(fw.act, fw.Wd[l], fw.emb, fw.xa, fw.ss_b))
    pk = peaks()
    by = fw.algorithmic_bytes()
    total = n * (by["dense_layer"] + by["attn_layer"]) + by["lmhead"] + by["tree"]
    frac = lambda b, us: round(b / (us * 1e-6) / 1e9 / pk["hbm"], 4)
    d, I, D = c["d"], c["inter"], c["D"]
    return {"workload": f"forward36: Qwen3-8B-shaped target, {n} layers (d={d}, {c['Hq']}/{c['Hkv']} heads, "
                        f"head_dim {D}, inter={I}), T={c['T']}, N={c['N']} (M={fw.R} rows), V={c['V']}",
            "rounds_per_s": round(1e6 / st["round"], 2),
            "stages_us": {k: round(v, 2) for k, v in st.items()},
            "round_bytes": total,
            "round_hbm_frac": frac(total, st["round"]),
            "layer_hbm_frac": frac(by["dense_layer"] + by["attn_layer"], st["layer"]),
            "qkv_hbm_frac": frac(d * (c["Hq"] + 2 * c["Hkv"]) * D * 2, st["qkv"]),
            "o_proj_hbm_frac": frac(c["Hq"] * D * d * 2, st["o_proj"]),
            "swiglu_hbm_frac": frac(2 * d * I * 2, st["swiglu"]),
            "down_proj_hbm_frac": frac(I * d * 2, st["down_proj"]),
            "gpu_launches_per_round": fw.launches_per_step(),
            "data": "synthetic, random-init weights, rows and K/V drawn on the device (seeded torch generator)"}


def mufu_peak():
    """ex2 per second of the special-function units: 16 per clock per SM
    (derived: 4 per clock per scheduler) x the SMs x the maximum SM clock."""
    import torch
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    return 16 * props.multi_processor_count * 2.07e9


def attn_roof_us(cfg, T, R, anc_sizes, pk):
    """Binding roof of one attention layer: max of HBM bytes, tensor flops and
    exponentials, each at its peak (us), and which one binds."""
    seen = sum(T + a for a in anc_sizes)  # keys each row attends to
    by = (T + R) * cfg["Hkv"] * cfg["D"] * 2 * 2 + 2 * R * cfg["Hq"] * cfg["D"] * 2
    fl = 4 * cfg["D"] * cfg["Hq"] * seen
    ex = cfg["Hq"] * seen
    t = {"hbm": by / (pk["hbm"] * 1e9) * 1e6, "tensor": fl / (pk["bf16"] * 1e12) * 1e6,
         "mufu": ex / mufu_peak() * 1e6}
    bind = max(t, key=t.get)
    return t[bind], bind, by


def run_entropy_sweep(dev, wl_W, reps=10):
    """Config 4 (secondary): tree build + 36 layers of tree attention at T =
    2048 for draft marginals of 0.3 / 1.5 / 4.0 nats and N in {31, 63, 127,
    255}, plus the LM head at M = N + 1 as an extra; each stage against its
    binding roof (HBM, tensor or exponentials)."""
    import torch
    import tree_verified_block_gb300 as g
    c = ENTROPY36
    pk = peaks()
    tg = torch.Generator(device=dev)
    tg.manual_seed(4000)
    n_max = max(c["N_set"]) + 1
    t_cap = c["T"] + n_max + 64
    rn = lambda *shape: torch.randn(*shape, generator=tg, device=dev).to(torch.bfloat16)
    k = [rn(c["Hkv"], t_cap, c["D"]) for _ in range(c["n_layers"])]
    v = [rn(c["Hkv"], t_cap, c["D"]) for _ in range(c["n_layers"])]
    q_all = [rn(n_max, c["Hq"], c["D"]) for _ in range(c["n_layers"])]
    h_all = rn(n_max, c["d"])
    t0 = torch.tensor([c["T"]], dtype=torch.int32, device=dev)
    t_len = t0.clone()
    root = torch.tensor([77], dtype=torch.int32, device=dev)
    layers = [g.KVLayer(kk, vv, t_len) for kk, vv in zip(k, v)]
    scale = c["D"] ** -0.5
    out = []
    for H in c["entropy"]:
        x = torch.from_numpy(W.draft_logits_entropy(c["L"], c["V"], H, seed=4100 + int(10 * H))).to(dev)
        for N in c["N_set"]:
            R = N + 1
            tree = g.Tree(N, c["L"], dev)
            ws_tree = g.workspace(g.build_tree_workspace_bytes(c["L"], c["V"], N), dev)
            ws_attn = g.workspace(g.tree_attention_workspace_bytes(R, c["Hq"], layers[0]), dev)
            ws_lm = g.workspace(g.lmhead_argmax_workspace_bytes(R, c["d"], c["V"], torch.bfloat16), dev)
            q = [qq[:R].contiguous() for qq in q_all]
            o = [torch.empty_like(qq) for qq in q]
            h = h_all[:R].contiguous()
            am = torch.empty(R, dtype=torch.int32, device=dev)
            gp = torch.empty(R, dtype=torch.float32, device=dev)
            mx = torch.empty(R, dtype=torch.float32, device=dev)

            def tree_fn():
                t_len.copy_(t0)
                g.build_tree(x, N, root, t_len, tree, ws_tree)
            tree_fn()
            torch.cuda.synchronize()
            depth = tree.depth.cpu().numpy()
            st = {"tree": graph_time_us(tree_fn, reps),
                  "attention_36": graph_time_us(
                      lambda: [g.tree_attention(q[l], layers[l], tree, scale, o[l], ws_attn)
                               for l in range(c["n_layers"])], reps),
                  "lmhead": graph_time_us(lambda: g.lmhead_argmax(h, wl_W, am, gp, mx, ws_lm), reps)}
            roof_us, bind, by = attn_roof_us(c, c["T"], R, [int(dd) + 1 for dd in depth], pk)
            per_layer = st["attention_36"] / c["n_layers"]
            lm_bytes = c["d"] * c["V"] * 2 + R * c["d"] * 2
            lm_roof = max(lm_bytes / (pk["hbm"] * 1e9), 2 * R * c["d"] * c["V"] / (pk["bf16"] * 1e12)) * 1e6
            out.append({"H": H, "N": N, "max_depth": int(depth.max()),
                        "tree_us": round(st["tree"], 2),
                        "tree_hbm_frac": round(c["L"] * c["V"] * 4 / (st["tree"] * 1e-6) / 1e9 / pk["hbm"], 4),
                        "attention_layer_us": round(per_layer, 2),
                        "attention_bound": bind,
                        "attention_frac_of_binding_roof": round(roof_us / per_layer, 4),
                        "lmhead_us": round(st["lmhead"], 2),
                        "lmhead_frac_of_binding_roof": round(lm_roof / st["lmhead"], 4),
                        "rounds_per_s_tree_attn": round(1e6 / (st["tree"] + st["attention_36"]), 1)})
    return {"workload": f"entropy36: T={c['T']}, L={c['L']}, V={c['V']}, {c['n_layers']} layers, "
                        f"draft entropy {list(c['entropy'])} nats x N {list(c['N_set'])}",
            "mufu_peak_ex2_per_s": mufu_peak(),
            "points": out,
            "data": "synthetic: draft logits calibrated to the entropy (seeded numpy), q/K/V/h drawn on the device"}


def run_verify1(dev, reps=20):
    """Config 2 (secondary): one layer at T = 1024, N = 31: tree build and
    tree attention."""
    import torch
    import tree_verified_block_gb300 as g
    c = VERIFY1
    pk = peaks()
    tg = torch.Generator(device=dev)
    tg.manual_seed(2000)
    R = c["N"] + 1
    t_cap = c["T"] + R + 64
    rn = lambda *shape: torch.randn(*shape, generator=tg, device=dev).to(torch.bfloat16)
    kv = g.KVLayer(rn(c["Hkv"], t_cap, c["D"]), rn(c["Hkv"], t_cap, c["D"]),
                   torch.tensor([c["T"]], dtype=torch.int32, device=dev))
    t0 = kv.t_len.clone()
    x = torch.from_numpy(W.draft_logits_planted(c["L"], c["V"], seed=2001)).to(dev)
    root = torch.tensor([5], dtype=torch.int32, device=dev)
    tree = g.Tree(c["N"], c["L"], dev)
    ws_tree = g.workspace(g.build_tree_workspace_bytes(c["L"], c["V"], c["N"]), dev)
    ws_attn = g.workspace(g.tree_attention_workspace_bytes(R, c["Hq"], kv), dev)
    q = rn(R, c["Hq"], c["D"])
    o = torch.empty_like(q)

    def tree_fn():
        kv.t_len.copy_(t0)
        g.build_tree(x, c["N"], root, kv.t_len, tree, ws_tree)
    tree_fn()
    torch.cuda.synchronize()
    depth = tree.depth.cpu().numpy()
    t_tree = graph_time_us(tree_fn, reps)
    t_attn = graph_time_us(lambda: g.tree_attention(q, kv, tree, c["D"] ** -0.5, o, ws_attn), reps)
    roof_us, bind, by = attn_roof_us(c, c["T"], R, [int(dd) + 1 for dd in depth], pk)
    return {"workload": f"verify1: 1 layer, T={c['T']}, N={c['N']}, L={c['L']}, V={c['V']}",
            "tree_us": round(t_tree, 2), "attention_us": round(t_attn, 2),
            "attention_bound": bind, "attention_frac_of_binding_roof": round(roof_us / t_attn, 4),
            "tree_hbm_frac": round(c["L"] * c["V"] * 4 / (t_tree * 1e-6) / 1e9 / pk["hbm"], 4),
            "data": "synthetic: planted-peak draft logits (seeded numpy), q/K/V drawn on the device"}


def run_case(args):
    """One workload alone, launched warmup + steps times, for profiler
    captures; prints its graph-timed duration. lmhead512: the LM head over 512
    stacked rows, [512, 4096] x [4096, 151936] (a few GB on the device).
    dense_layer: the four projections of one Qwen3-8B-shaped layer at M = 64
    (386 MB of weights). forward36: the whole forward36 round (~16 GB).
    Inputs drawn on the device."""
    import torch
    import tree_verified_block_gb300 as g
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.case in ("dense_layer", "forward36"):
        cfg = FORWARD36 if args.case == "forward36" else dict(FORWARD36, n_layers=1, V=16384)
        fw = ForwardWorkload(cfg, dev)
        c = fw.cfg
        if args.case == "forward36":
            fn = fw.step
        else:
            def fn():
                g.dense_qkv(fw.emb, fw.Wqkv[0], c["Hq"], fw.ss0, None, None, c["eps"], fw.tree.pos_id,
                            c["rope_theta"], fw.q, fw.layers[0])
                g.dense_residual(fw.att.view(fw.R, -1), fw.Wo[0], fw.emb, fw.xa, fw.ss_a)
                g.dense_swiglu(fw.xa, fw.Wg[0], fw.Wu[0], fw.ss_a, c["eps"], fw.act)
                g.dense_residual(fw.act, fw.Wd[0], fw.emb, fw.xa, fw.ss_b)
            fw.step()  # tree, input sums of squares, caches
        for _ in range(args.warmup + args.steps):
            fn()
        torch.cuda.synchronize()
        us = graph_time_us(fn, 10)
        by = fw.algorithmic_bytes()
        b = by["dense_layer"] if args.case == "dense_layer" else (
            c["n_layers"] * (by["dense_layer"] + by["attn_layer"]) + by["lmhead"] + by["tree"])
        print(json.dumps({"case": args.case, "us": round(us, 2),
                          "hbm_frac": round(b / (us * 1e-6) / 1e9 / peaks()["hbm"], 4)}), flush=True)
        return
    if args.case in ("attn255", "attn_ragged8"):
        run_attn_case(args, dev)
        return
    if args.case in ("tree63", "tree255"):
        run_tree_case(args, dev)
        return
    M, d, V = 512, 4096, 151936
    tg = torch.Generator(device=dev)
    tg.manual_seed(7)
    h = torch.randn(M, d, generator=tg, device=dev).to(torch.bfloat16)
    Wt = (torch.randn(d, V, generator=tg, device=dev) * 0.02).to(torch.bfloat16)
    am = torch.empty(M, dtype=torch.int32, device=dev)
    gap = torch.empty(M, dtype=torch.float32, device=dev)
    mx = torch.empty(M, dtype=torch.float32, device=dev)
    ws = g.workspace(g.lmhead_argmax_workspace_bytes(M, d, V, torch.bfloat16), dev)
    ent = torch.empty(M, dtype=torch.float32, device=dev)
    pos = torch.arange(M, dtype=torch.int32, device=dev) % 64 + 4096
    seq = torch.arange(M, dtype=torch.int32, device=dev) // 64
    fn = {"lmhead512": lambda: g.lmhead_argmax(h, Wt, am, gap, mx, ws),
          "lmhead512_entropy": lambda: g.lmhead_argmax_entropy(h, Wt, am, gap, mx, ent, ws),
          "lmhead512_sample": lambda: g.lmhead_sample(h, Wt, 1.0, 5, pos, seq, am, gap, ws)}[args.case]
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize()
    us = graph_time_us(fn, 10)
    tf = 2 * M * d * V / (us * 1e-6) / 1e12
    pk = peaks()
    print(json.dumps({"case": args.case, "us": round(us, 2), "tflops": round(tf, 1),
                      "tensor_frac": round(tf / pk["bf16"], 4)}), flush=True)


def run_gpu(args):
    import torch
    import tree_verified_block_gb300 as g
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g.lib()
    cfg = SMALL if args.workload == "small" else FULL36
    wl = Workload(cfg, dev, seed=3000, keep_host=False)
    torch.cuda.synchronize()
    # warm-up, then capture one round in a CUDA graph
    for _ in range(max(1, args.warmup)):
        wl.step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        wl.step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        start.record(stream)
        for _ in range(args.steps):
            graph.replay()
        end.record(stream)
        torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    ms_per_step = ms / args.steps
    value = args.steps / (ms / 1e3)
    # spread of single steps (each replay between its own events, after the timed region)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(100)]
    for a_, b_ in evs:
        a_.record(stream)
        graph.replay()
        b_.record(stream)
    torch.cuda.synchronize()
    per = sorted(a_.elapsed_time(b_) * 1e3 for a_, b_ in evs)
    spread = {"p10": round(per[10], 2), "p50": round(per[50], 2), "p90": round(per[90], 2), "n": len(per)}

    # per-stage times (eager, events on the launching stream)
    st = stage_times(wl)
    bytes_ = wl.algorithmic_bytes()
    pk = peaks()
    attn_total = st["attention_36"]
    dominant = "lmhead" if st["lmhead"] >= attn_total else "attention"
    kernel = "glance_lmhead_argmax" if dominant == "lmhead" else "glance_tree_attention"
    if dominant == "lmhead":
        dur = st["lmhead"]
        achieved = bytes_["lmhead"] / (dur * 1e-6) / 1e9
    else:
        # per launch in the round's 36-layer chain (each launch's prologue
        # overlaps the previous layer's tail, as in the timed region)
        dur = attn_total / cfg["n_layers"]
        achieved = bytes_["attn_layer"] / (dur * 1e-6) / 1e9
    roofline = {"bound": "hbm", "kernel": kernel,
                "achieved": round(achieved, 1), "peak": pk["hbm"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm"], 4), "traffic": profiled_traffic(kernel),
                "algorithmic_bytes": bytes_["lmhead" if dominant == "lmhead" else "attn_layer"],
                "peak_source": pk["src"] + " copy (burst; the kernel's launches are timed without the other stages)",
                "launch_us": round(dur, 2)}
    lm_tflops = wl.flops()["lmhead"] / (st["lmhead"] * 1e-6) / 1e12
    stages = {k: round(v, 2) for k, v in st.items()}
    stages["lmhead_tensor_tflops"] = round(lm_tflops, 1)
    stages["lmhead_tensor_frac_of_peak"] = round(lm_tflops / pk["bf16"], 4)
    stages["attention_per_layer_in_chain"] = round(attn_total / cfg["n_layers"], 2)
    stages["attention_layer_hbm_frac"] = round(bytes_["attn_layer"] * cfg["n_layers"] / (attn_total * 1e-6) / 1e9 / pk["hbm"], 4)
    stages["lmhead_hbm_frac"] = round(bytes_["lmhead"] / (st["lmhead"] * 1e-6) / 1e9 / pk["hbm"], 4)
    stages["tree_hbm_frac"] = round(bytes_["tree"] / (st["tree"] * 1e-6) / 1e9 / pk["hbm"], 4)

    e2e = run_e2e(wl, args.steps)
    batched = run_batched(dev) if args.batched else None
    forward = run_forward(dev) if args.forward else None
    sweep = run_entropy_sweep(dev, wl.W) if args.sweep else None
    verify1 = run_verify1(dev) if args.sweep else None
    code, text = g.device_status()
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "rounds/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(cfg),
        "roofline": roofline,
        "stages_us": stages,
        "step_us_percentiles": spread,
        "e2e": e2e,
        "gpu_launches": wl.launches_per_step() * args.steps,
        "clocks": clk.summary(),
        "device_status": code,
    }
    if batched is not None:
        out["ragged8"] = batched
    if forward is not None:
        out["forward36"] = forward
    if sweep is not None:
        out["entropy36"] = sweep
        out["verify1"] = verify1
    if args.cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg)
    print(json.dumps(out), flush=True)


def run_e2e(wl, steps):
    """Same metric through the public Python API with host buffers: the step's
    inputs (draft logits, per-layer q, the tree rows' K/V, h) come from one
    pinned host buffer and the round's result is read back, inside the timed
    region. The step — one host-to-device copy of that buffer into a device
    staging buffer (the round reads logits, q and h there in place; the tree
    rows' K/V are copied on into the caches), the round's calls and the
    read-back — is captured once in a CUDA graph, as a serving loop would,
    and each step replays it and waits for the result on the host. The same
    step with the inputs copied tensor by tensor and every call launched from
    Python is reported beside it (eager_value)."""
    import torch
    c = wl.cfg
    R, T = wl.R, c["T"]
    # pinned host image of the step's inputs: logits | q x 36 | h | tree rows' K/V
    # [36][2][Hkv][R][D] (the layout glance_kv_write_rows scatters from)
    kv_rows = torch.stack([torch.stack([k[:, T:T + R], v[:, T:T + R]]) for k, v in zip(wl.k, wl.v)])
    parts = [wl.x_dev.view(torch.uint8).reshape(-1)] + [q.view(torch.uint8).reshape(-1) for q in wl.q] + \
            [wl.h.view(torch.uint8).reshape(-1), kv_rows.contiguous().view(torch.uint8).reshape(-1)]
    sizes = [int(t.numel()) for t in parts]
    offs = np.cumsum([0] + sizes)
    host = torch.empty(int(offs[-1]), dtype=torch.uint8, pin_memory=True)
    for t, o in zip(parts, offs[:-1]):
        host[int(o):int(o) + t.numel()].copy_(t.cpu())
    stage = torch.empty_like(host, device=wl.x_dev.device)
    view = lambda i, like: stage[int(offs[i]):int(offs[i + 1])].view(like.dtype).view(like.shape)
    n = c["n_layers"]
    x_s = view(0, wl.x_dev)
    q_s = [view(1 + l, wl.q[l]) for l in range(n)]
    h_s = view(1 + n, wl.h)
    kv_s = view(2 + n, kv_rows)
    res = torch.empty(2 + c["L"], dtype=torch.int32, pin_memory=True)
    h2d = int(offs[-1])
    d2h = res.numel() * 4
    saved = (wl.x_dev, wl.q, wl.h)
    kv_e = torch.empty_like(kv_rows)

    def readback():
        res[0:1].copy_(wl.n_acc, non_blocking=True)
        res[1:2].copy_(wl.new_root, non_blocking=True)
        res[2:].copy_(wl.acc_tok, non_blocking=True)

    def staged():
        stage.copy_(host, non_blocking=True)
        wl.g.kv_write_rows(kv_s, wl.layers, R)
        wl.step()
        readback()

    def eager():
        wl.x_dev.copy_(host[int(offs[0]):int(offs[1])].view(torch.float32).view(wl.x_dev.shape), non_blocking=True)
        for l in range(n):
            wl.q[l].copy_(host[int(offs[1 + l]):int(offs[2 + l])].view(wl.q[l].dtype).view(wl.q[l].shape),
                          non_blocking=True)
        kv_e.copy_(host[int(offs[2 + n]):int(offs[3 + n])].view(torch.bfloat16).view(kv_rows.shape),
                   non_blocking=True)
        wl.g.kv_write_rows(kv_e, wl.layers, R)
        wl.h.copy_(host[int(offs[1 + n]):int(offs[2 + n])].view(torch.bfloat16).view(wl.h.shape), non_blocking=True)
        wl.step()
        readback()
        torch.cuda.current_stream().synchronize()

    for _ in range(2):
        eager()
    t0 = time.perf_counter()
    n_eager = max(1, steps // 4)
    for _ in range(n_eager):
        eager()
    eager_rate = n_eager / (time.perf_counter() - t0)
    # the round reads its logits, q and h in the staging buffer
    wl.x_dev, wl.q, wl.h = x_s, q_s, h_s
    try:
        staged()
        torch.cuda.current_stream().synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            staged()
        for _ in range(3):
            graph.replay()
            torch.cuda.current_stream().synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            graph.replay()
            torch.cuda.current_stream().synchronize()
            _ = int(res[0])  # the host reads the result
        serial_rate = steps / (time.perf_counter() - t0)
    finally:
        wl.x_dev, wl.q, wl.h = saved

    # Pipelined: two staging buffers and two captured rounds; step i + 1's
    # host-to-device copy (on a copy stream) overlaps step i's round, and the
    # host reads each step's result as soon as that step is done. Every step
    # still copies its inputs and returns its result inside the timed region.
    dev = wl.x_dev.device
    stages = [stage, torch.empty_like(host, device=dev)]
    results = [res, torch.empty(res.shape, dtype=res.dtype, pin_memory=True)]
    graphs = []
    main, cs = torch.cuda.current_stream(), torch.cuda.Stream(device=dev)
    for b in range(2):
        vw = lambda i, like, b=b: stages[b][int(offs[i]):int(offs[i + 1])].view(like.dtype).view(like.shape)
        xb, qb, hb = vw(0, saved[0]), [vw(1 + l, saved[1][l]) for l in range(n)], vw(1 + n, saved[2])
        kvb = vw(2 + n, kv_rows)
        wl.x_dev, wl.q, wl.h = xb, qb, hb
        rb = results[b]

        def body(kvb=kvb, rb=rb):
            wl.g.kv_write_rows(kvb, wl.layers, R)
            wl.step()
            rb[0:1].copy_(wl.n_acc, non_blocking=True)
            rb[1:2].copy_(wl.new_root, non_blocking=True)
            rb[2:].copy_(wl.acc_tok, non_blocking=True)
        try:
            stages[b].copy_(host)
            body()
            torch.cuda.synchronize()
            gph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gph):
                body()
            graphs.append(gph)
        finally:
            wl.x_dev, wl.q, wl.h = saved
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]

    def run(n_steps):
        for i in range(n_steps):
            b = i & 1
            if i >= 2:
                cs.wait_event(done[b])  # step i - 2 is done with this staging buffer
            with torch.cuda.stream(cs):
                stages[b].copy_(host, non_blocking=True)
                ready[b].record(cs)
            main.wait_event(ready[b])
            graphs[b].replay()
            done[b].record(main)
            if i >= 1:
                done[b ^ 1].synchronize()
                _ = int(results[b ^ 1][0])  # the host reads step i - 1's result
        done[(n_steps - 1) & 1].synchronize()
        _ = int(results[(n_steps - 1) & 1][0])

    run(4)
    t0 = time.perf_counter()
    run(steps)
    dt = time.perf_counter() - t0
    return {"value": round(steps / dt, 2), "unit": "rounds/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": int(d2h), "serial_value": round(serial_rate, 2),
            "eager_value": round(eager_rate, 2),
            "note": "each step: one pinned host->device copy of its inputs (copy stream), then one "
                    "glance_kv_write_rows launch puts the tree rows' K/V of all layers into the caches, "
                    "the round and the read-back (one CUDA graph); step i + 1's copy overlaps step i's "
                    "round, the host reads every result. serial_value: copy, round and read-back back to "
                    "back; eager_value: inputs copied tensor by tensor and every call launched from Python"}


# ------------------------------------------------------------------ oracle

# One bounded oracle step, shared by the GPU line's cpu_baseline and the
# reference arm, so that both time the same sample with the same scaling.
ORACLE_SAMPLE = dict(l_sub=3, rows=8, kv_heads=1, layers=1, lm_cols=148)


def oracle_sample_text(cfg):
    o = ORACLE_SAMPLE
    return (f"per step: tree build on {o['l_sub']} of {cfg['L']} offsets (x {cfg['L'] / o['l_sub']:g}); "
            f"attention of {o['rows']} of {cfg['N'] + 1} rows x {o['kv_heads']} of {cfg['Hkv']} kv heads x "
            f"{o['layers']} of {cfg['n_layers']} layers; LM head over {o['lm_cols']} of {cfg['V']} columns; "
            f"walk + commit on {o['layers']} of {cfg['n_layers']} layers; each stage's time scaled by "
            f"its sampled fraction to a full round")


class HostInputs:
    """Host-only inputs of the oracle step (no GPU): the full draft logits,
    one layer of q/K/V, the LM head's h and ORACLE_SAMPLE['lm_cols'] columns
    of W, and the full tree built once."""

    def __init__(self, cfg, seed=3000):
        from oracle.tree import build_tree as o_build
        gen = W.rng(seed)
        R = cfg["N"] + 1
        t_cap = cfg["T"] + R + 64
        self.x = W.draft_logits_planted(cfg["L"], cfg["V"], seed=seed + 1)
        self.q_bits = [W.normal_bf16(gen, (R, cfg["Hq"], cfg["D"]))]
        self.k_bits = [W.normal_bf16(gen, (cfg["Hkv"], t_cap, cfg["D"]))]
        self.v_bits = [W.normal_bf16(gen, (cfg["Hkv"], t_cap, cfg["D"]))]
        self.W_bits = W.normal_bf16(gen, (cfg["d"], ORACLE_SAMPLE["lm_cols"]), std=0.02)
        self.h_bits = W.normal_bf16(gen, (R, cfg["d"]))
        self.tree = o_build(self.x.astype(np.float64), cfg["N"], 7, cfg["T"])


def oracle_step(cfg, src, root=7):
    """One bounded oracle step: each stage of the round on the slice that
    ORACLE_SAMPLE names, its time scaled by the sampled fraction to the full
    stage. Returns (scaled seconds of a full round, per-stage detail, wall
    seconds the step took)."""
    from oracle.attention import tree_attention as o_attn
    from oracle.bf16 import bf16_bits_to_f64
    from oracle.lmhead import lmhead_argmax as o_lmhead
    from oracle.tree import build_tree as o_build
    from oracle.walk import commit as o_commit
    from oracle.walk import walk as o_walk
    o = ORACLE_SAMPLE
    T, R, G = cfg["T"], cfg["N"] + 1, cfg["Hq"] // cfg["Hkv"]
    t = {}
    w0 = time.perf_counter()
    t0 = time.perf_counter()
    o_build(src.x[:o["l_sub"]].astype(np.float64), cfg["N"], root, T)
    t["tree"] = (time.perf_counter() - t0) * cfg["L"] / o["l_sub"]
    tree = src.tree  # the full tree (built once) for the stages below
    t0 = time.perf_counter()
    o_attn(bf16_bits_to_f64(src.q_bits[0][:o["rows"], :G * o["kv_heads"]]),
           bf16_bits_to_f64(src.k_bits[0][:o["kv_heads"], :T + R]),
           bf16_bits_to_f64(src.v_bits[0][:o["kv_heads"], :T + R]), T, tree["anc"][:o["rows"]],
           cfg["D"] ** -0.5)
    t["attention"] = ((time.perf_counter() - t0) * (R / o["rows"]) * (cfg["Hkv"] / o["kv_heads"])
                      * cfg["n_layers"] / o["layers"])
    t0 = time.perf_counter()
    arg, _, _ = o_lmhead(bf16_bits_to_f64(src.h_bits), bf16_bits_to_f64(src.W_bits))
    t["lmhead"] = (time.perf_counter() - t0) * cfg["V"] / src.W_bits.shape[1]
    t0 = time.perf_counter()
    a, path, _, _ = o_walk(tree, arg, cfg["L"])
    o_commit(src.k_bits[0].copy(), src.v_bits[0].copy(), T, path)
    t["commit"] = (time.perf_counter() - t0) * cfg["n_layers"] / o["layers"]
    return sum(t.values()), t, time.perf_counter() - w0


def oracle_summary(cfg, totals, parts, walls):
    sec = statistics.median(totals)
    return {"value": round(1.0 / sec, 5), "unit": "rounds/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle", "sample": oracle_sample_text(cfg), "steps_timed": len(totals),
            "wall_seconds_per_step": round(statistics.median(walls), 4),
            "rounds_per_step": round(statistics.median(walls) / sec, 8),
            "stage_seconds_full_round": {k: round(statistics.median(p[k] for p in parts), 3)
                                         for k in parts[0]}}


def cpu_baseline(cfg, seconds=10.0):
    """The oracle as it stands on the host cores: the same bounded step as
    the reference arm, repeated for about `seconds` (at least 3 steps);
    value = 1 / the median scaled round."""
    src = HostInputs(cfg)
    oracle_step(cfg, src)
    totals, parts, walls = [], [], []
    t0 = time.perf_counter()
    while len(totals) < 3 or time.perf_counter() - t0 < seconds:
        tt, pp, ww = oracle_step(cfg, src)
        totals.append(tt)
        parts.append(pp)
        walls.append(ww)
    return oracle_summary(cfg, totals, parts, walls)


def run_reference(args):
    """The oracle (the reference arm of this build), as it stands, on the
    host cores: every step is the bounded oracle step (about 0.1 s on a GB300
    host), scaled to a full round, so that any --steps K ends in a few
    minutes. ms_per_step is the wall time a step took; rounds_per_step is the
    fraction of a round it covers, so value = rounds_per_step / step time."""
    cfg = SMALL if args.workload == "small" else FULL36
    src = HostInputs(cfg)
    for _ in range(args.warmup):
        oracle_step(cfg, src)
    totals, parts, walls = [], [], []
    for _ in range(args.steps):
        tt, pp, ww = oracle_step(cfg, src)
        totals.append(tt)
        parts.append(pp)
        walls.append(ww)
    base = oracle_summary(cfg, totals, parts, walls)
    value = base["value"]
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rounds/s",
           "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(statistics.median(walls) * 1e3, 2),
           "rounds_per_step": base["rounds_per_step"],
           "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": workload_config(cfg), "cpu_baseline": base,
           "e2e": {"value": value, "unit": "rounds/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_tree_case(args, dev):
    """The draft-to-tree build alone, for profiler captures: tree63 = the
    full36 draft marginals (15 x 151936 planted logits, N = 63); tree255 =
    4.0-nat marginals at N = 255 (the entropy sweep's bushiest tree).
    Inputs drawn on the host from seeded generators and copied once."""
    import torch
    import tree_verified_block_gb300 as g
    L, V = FULL36["L"], FULL36["V"]
    if args.case == "tree63":
        N, x = 63, W.draft_logits_planted(L, V, seed=3001)
    else:
        N, x = 255, W.draft_logits_entropy(L, V, 4.0, seed=4140)
    xd = torch.from_numpy(x).to(dev)
    tree = g.Tree(N, L, dev)
    ws = g.workspace(g.build_tree_workspace_bytes(L, V, N), dev)
    t_len = torch.tensor([FULL36["T"]], dtype=torch.int32, device=dev)
    root = torch.tensor([1234], dtype=torch.int32, device=dev)
    fn = lambda: g.build_tree(xd, N, root, t_len, tree, ws)
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize()
    us = graph_time_us(fn, 20)
    print(json.dumps({"case": args.case, "us": round(us, 2)}), flush=True)


def run_attn_case(args, dev):
    """One tree-attention layer alone, for profiler captures: attn255 = one
    layer at T = 2048, N = 255 (1024 query rows per kv head: tensor / MUFU
    bound); attn_ragged8 = one batched layer of the ragged8 batch (8 requests,
    T ~ U{512..8192}, N = 63). Inputs drawn on the device."""
    import torch
    import tree_verified_block_gb300 as g
    tg = torch.Generator(device=dev)
    tg.manual_seed(11)
    rn = lambda *shape: torch.randn(*shape, generator=tg, device=dev).to(torch.bfloat16)
    scale = 128 ** -0.5
    if args.case == "attn255":
        c = dict(ENTROPY36, N=255)
        R = c["N"] + 1
        t_len = torch.tensor([c["T"]], dtype=torch.int32, device=dev)
        layer = g.KVLayer(rn(c["Hkv"], c["T"] + R + 64, c["D"]), rn(c["Hkv"], c["T"] + R + 64, c["D"]), t_len)
        x = torch.from_numpy(W.draft_logits_entropy(c["L"], c["V"], 4.0, seed=4140)).to(dev)
        tree = g.Tree(c["N"], c["L"], dev)
        g.build_tree(x, c["N"], torch.tensor([77], dtype=torch.int32, device=dev), t_len, tree,
                     g.workspace(g.build_tree_workspace_bytes(c["L"], c["V"], c["N"]), dev))
        q = rn(R, c["Hq"], c["D"])
        o = torch.empty_like(q)
        ws = g.workspace(g.tree_attention_workspace_bytes(R, c["Hq"], layer), dev)
        fn = lambda: g.tree_attention(q, layer, tree, scale, o, ws)
        flops = sum(4 * c["D"] * c["Hq"] * (c["T"] + int(bin(int(w)).count("1")))
                    for w in tree.to_host()["anc"].reshape(R, -1)[:, 0])
    else:
        bw = BatchedWorkload(RAGGED8, dev, host=False, n_layers=1)
        fn = lambda: g.tree_attention_batched(bw.q[0], bw.layers[0], bw.trees, scale, bw.out[0], bw.ws_attn)
        flops = None
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize()
    us = graph_time_us(fn, 10)
    out = {"case": args.case, "us": round(us, 2)}
    if flops:
        out["tflops"] = round(flops / (us * 1e-6) / 1e12, 1)
    print(json.dumps(out), flush=True)


def run_unavailable(args):
    """More than one GPU: the path is per request (one GPU per request, no
    exchange), so this benchmark runs on one GPU only."""
    if os.environ.get("RANK", "0") != "0":
        return
    print(json.dumps({"impl": args.impl, "metric": METRIC, "n_gpus": args.gpus,
                      "unavailable": "single-GPU benchmark: a verify round runs on one GPU; "
                                     "more GPUs would only run independent replicas"}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="glance", choices=["glance", "reference"])
    ap.add_argument("--workload", default="full36", choices=["full36", "small"])
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--case", default=None, choices=["lmhead512", "lmhead512_entropy", "lmhead512_sample",
                                                     "attn255", "attn_ragged8", "dense_layer", "forward36",
                                                     "tree63", "tree255"],
                    help="run one kernel alone on a small case (for profiler captures)")
    ap.add_argument("--no-sweep", dest="sweep", action="store_false",
                    help="skip the entropy36 sweep and the verify1 single-layer case")
    ap.add_argument("--no-forward", dest="forward", action="store_false",
                    help="skip the forward36 secondary measurement (verify forward with the dense layers)")
    ap.add_argument("--no-batched", dest="batched", action="store_false",
                    help="skip the secondary ragged8 batched-round measurement")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus != 1:
        run_unavailable(args)
    elif args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
