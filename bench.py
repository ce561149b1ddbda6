#!/usr/bin/env python
"""Benchmark of the bit-exact fixed-order FP32 hot path on GB300.

One step = one pass of every operation of the path over one batch of the
162M-decoder workloads (shapes from the "MojoLearn 162M" model card, table
"Compared with GPT-3 Small"; 8,192 tokens = 4 x 2,048):
  RMSNorm 8192 x 768 -> forward GEMMs (QKV 768x2304, out 768x768, SwiGLU gate and
  up 768x2048, down 2048x768, LM head 768x50257 with the [out, in] weight) ->
  softmax cross-entropy over 8192 x 50257 logits (loss, mean, dlogits) ->
  RMSNorm backward 8192 x 768 (dx, dgain) ->
  weight-gradient GEMMs X^T dY over the 8,192 tokens (768x2304, 2048x768) ->
  fixed-order sum of 64 gathered shard gradients of the 768x2304 weight ->
  one pre-norm decoder block forward (RMSNorm, QKV, RoPE, causal attention,
  out projection, residual, RMSNorm, SwiGLU, down projection, residual) ->
  one training step of the byte-level LM (16 x 128 tokens, two blocks of 64:
  forward, backward, AdamW) ->
  the 12-layer 162M decoder's forward with its loss (4 x 2048 tokens) ->
  AdamW over 162,147,840 parameters.
Inputs are synthetic and seeded (bitwise_reproducible_fp32_gb300.inputs).

value: fixed-order FP32 GEMM TFLOP/s = the step's GEMM FLOPs / the GEMM kernels'
device time (CUDA events on the launching stream). The reduce/AdamW rates are
under "ops". L2 is flushed (a 512 MB write, then a 512 MB read of another buffer) before every timed step.

--impl reference times the CPU oracle (the path's only reference
implementation) on a bounded sample of the same workload, on this host's cores.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bitwise_reproducible_fp32_gb300 import inputs  # noqa: E402

METRIC = ("bit-exact fixed-order FP32 GEMM TFLOP/s (% FP32 FMA peak); "
          "reduce/AdamW GB/s")
WORKLOAD = ("162M-decoder FP32 step: RMSNorm 8192x768 (once, then 16 times over distinct "
            "inputs), forward GEMMs "
            "(8192 tokens; 768x2304, 768x768, 2x 768x2048, 2048x768, LM head "
            "768x50257), softmax cross-entropy 8192x50257 with dlogits and mean, "
            "RMSNorm backward 8192x768 (dx, dgain; once, then 8 times over distinct inputs), "
            "dW GEMMs over 8192 tokens "
            "(768x2304, 2048x768), fixed-order sum of 64 shard gradients of the "
            "768x2304 weight, one decoder block forward (4x2048 tokens, RoPE, causal "
            "attention 12x64, SwiGLU), one byte-level LM training step (16x128 tokens, "
            "2 blocks of 64), the 12-layer 162M decoder forward with loss (4x2048 "
            "tokens), the 162M model's training step (forward, backward, AdamW; 4x2048 "
            "tokens), AdamW 162,147,840 params")
SM_COUNT = 152
FP32_LANES_PER_SM = 128


def fp32_peak_tflops(sm_mhz: float, sms: int = SM_COUNT) -> float:
    """CUDA-core FP32 FMA peak: SMs x 128 lanes x 2 flops x clock."""
    return sms * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "sm_max_mhz": 2070.0}, "fallback"


# ------------------------------------------------------------------ workload
def gemm_list():
    fwd = inputs.gemm_cfg3()
    dw = inputs.dw_cfg5()
    return fwd, dw


def gemm_dims(p):
    A, B = p["A"], p["B"]
    M = A.shape[1] if p["transA"] else A.shape[0]
    K = A.shape[0] if p["transA"] else A.shape[1]
    N = B.shape[0] if p["transB"] else B.shape[1]
    return M, N, K


# launches of the RMSNorm forward and backward rows timed back to back
RMS_RUN = 16
RMSB_RUN = 8


# the end-to-end leg's LM head row blocks and AdamW element blocks
E2E_LM_ROWS = 1024
E2E_ADAMW_BLOCKS = 8


def hbm_row(nbytes, seconds, hbm, **extra):
    """Rate of an HBM-bound row: algorithmic bytes over seconds a launch."""
    return {"gbs": nbytes / seconds / 1e9, "frac_hbm": nbytes / seconds / 1e9 / hbm,
            "ms": seconds * 1e3, **extra}


def bytes_rmsnorm(rows, D):
    return rows * D * 8 + D * 4 + rows * 4


def bytes_rmsnorm_bwd(rows, D):
    # read x, dy; write dx; gain, inv_rms, dgain
    return 12 * rows * D + 8 * D + 4 * rows


def bytes_shardsum(nshards, n):
    return 4 * nshards * n + 4 * n


def bytes_xent(rows, V, dlogits=True):
    return rows * V * 4 * (2 if dlogits else 1) + rows * 12


def bytes_adamw(n):
    return n * 28


# ------------------------------------------------------------------ ranks
def input_digests(groups):
    """SHA-256 of each workload's input bytes, the arrays taken in the listed
    order (shape and dtype included), so a result names exactly the inputs it
    was measured on. groups: {name: [arrays]}."""
    import hashlib
    out = {}
    for name, arrays in groups.items():
        h = hashlib.sha256()
        for a in arrays:
            a = np.ascontiguousarray(a)
            h.update(f"{a.dtype.str}{a.shape}".encode())
            h.update(memoryview(a).cast("B"))
        out[name] = h.hexdigest()
    return out


def workload_arrays(fwd, dw, r4, rb, sg, bc, bl, dm, aw):
    """The input arrays of each bench workload, in draw order."""
    def model(c):
        arrs = [c["tokens"], c["labels"], c["emb"]]
        for b in c["blocks"]:
            arrs += [b[k] for k in ("g1", "W_qkv", "W_o", "g2", "W_gate", "W_up", "W_down")]
        return arrs + [c["head"]]
    return {
        "gemm_forward": [a for p in fwd for a in (p["A"], p["B"])],
        "gemm_dw": [a for p in dw for a in (p["A"], p["B"])],
        "rowops": [r4[k] for k in ("x", "gain", "logits", "labels")],
        "rmsnorm_bwd_dy": [rb["dy"]],
        "shard_grads": [sg],
        "block": [bc[k] for k in ("x", "g1", "W_qkv", "W_o", "g2", "W_gate", "W_up", "W_down")],
        "byte_lm": model(bl),
        "decoder_162m": model(dm),
        "adamw": [aw[k] for k in ("p", "g", "m", "v")],
    }


def max_over_ranks(values, device):
    """Element-wise max of per-rank timings (every rank gets the result). The
    only collective of the benchmark: the path itself has no exchange, each
    rank runs an independent replica of the step."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def replica_throughput(work_per_rank, world, slowest_ms):
    """Whole-job rate: the work all replicas did over the slowest one's time."""
    return work_per_rank * world / (slowest_ms / 1e3)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # the raw samples (the JSON line carries their summary); the directory
        # can be redirected with DET_BENCH_OUT
        out = os.environ.get("DET_BENCH_OUT", os.path.join(ROOT, "bench_out"))
        self.path = os.path.join(out, f"clocks_gpu{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() in ("active", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["smax"] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ GPU arm
def run_ours(args, rank, world, local_rank):
    import torch

    from bitwise_reproducible_fp32_gb300 import build as libbuild
    from bitwise_reproducible_fp32_gb300 import detlib

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    libbuild.build()
    detlib.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    t_setup = time.time()
    fwd, dw = gemm_list()
    r4 = inputs.rowops_cfg4()
    rb = inputs.rmsnorm_bwd_cfg4()
    sg = inputs.shard_grads()
    bc = inputs.block_cfg()
    bl = inputs.byte_lm_cfg2()
    aw = inputs.adamw_cfg5()
    host = dict(fwd=fwd, dw=dw, r4=r4, rb=rb, sg=sg, bc=bc, aw=aw)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    # device-resident inputs (shared tensors uploaded once)
    cache = {}

    def dev_of(a):
        k = id(a)
        if k not in cache:
            cache[k] = up(a)
        return cache[k]

    g_fwd = [(p, dev_of(p["A"]), dev_of(p["B"])) for p in fwd]
    g_dw = [(p, dev_of(p["A"]), dev_of(p["B"])) for p in dw]
    c_fwd = [torch.empty(gemm_dims(p)[:2], dtype=torch.float32, device=dev) for p in fwd]
    c_dw = [torch.empty(gemm_dims(p)[:2], dtype=torch.float32, device=dev) for p in dw]
    # caller-owned split-K workspaces (None where the library needs none)
    # the gate and up projections read the same activations: one group (one
    # transposed copy of X, one grid for both), as the decoder block runs them
    names = [p["name"] for p in fwd]
    gu = (names.index("swiglu_gate"), names.index("swiglu_up"))
    gu_probs = [dict(A=g_fwd[i][1], B=g_fwd[i][2], C=c_fwd[i]) for i in gu]
    ws_gu = detlib.gemm_group_workspace(gu_probs, device=dev)
    ws_fwd = [None if i in gu else
              detlib.gemm_workspace(*gemm_dims(p), p["transA"], p["transB"], device=dev)
              for i, p in enumerate(fwd)]
    # the two weight-gradient GEMMs as one group: each has its own CTAs in one
    # grid, so the grid's last round is filled from both
    dw_probs = [dict(A=A, B=B, C=c_dw[i], transA=p["transA"], transB=p["transB"])
                for i, (p, A, B) in enumerate(g_dw)]
    ws_dw = detlib.gemm_group_workspace(dw_probs, device=dev)
    x4, gain4 = up(r4["x"]), up(r4["gain"])
    y4 = torch.empty_like(x4)
    inv4 = torch.empty(x4.shape[0], dtype=torch.float32, device=dev)
    logits, labels = up(r4["logits"]), up(r4["labels"])
    loss = torch.empty(logits.shape[0], dtype=torch.float32, device=dev)
    lmean = torch.empty(1, dtype=torch.float32, device=dev)
    dlog = torch.empty_like(logits)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dy4 = up(rb["dy"])
    dx4 = torch.empty_like(dy4)
    dgain4 = torch.empty(x4.shape[1], dtype=torch.float32, device=dev)
    ws_rb = torch.empty((detlib.detrmsnorm_bwd_workspace_bytes(*x4.shape) + 3) // 4,
                        dtype=torch.float32, device=dev)
    # RMSNorm runs 12 us and its backward 25 us: besides one launch each, the
    # step times a run of launches over distinct copies of the inputs (805 MB
    # and 604 MB in all, several times the L2), so every launch reads from
    # HBM and the per-launch time is the run's time over its launches
    rms_runs = [(x4.clone(), torch.empty_like(x4), torch.empty_like(inv4))
                for _ in range(RMS_RUN)]
    rmsb_runs = [(x4.clone(), dy4.clone(), torch.empty_like(dx4), torch.empty_like(dgain4))
                 for _ in range(RMSB_RUN)]
    shards = up(sg)
    gsum = torch.empty(sg.shape[1], dtype=torch.float32, device=dev)
    from bitwise_reproducible_fp32_gb300 import block as blockmod
    blk = blockmod.Block(bc["batch"], bc["seq"], bc["x"].shape[1], bc["W_gate"].shape[1],
                         inputs.N_HEADS, dev)
    bx = up(bc["x"])
    bw = {k: up(bc[k]) for k in ("g1", "W_qkv", "W_o", "g2", "W_gate", "W_up", "W_down")}
    from bitwise_reproducible_fp32_gb300 import byte_lm
    bld = dict(bl)
    bld["tokens"] = torch.from_numpy(bl["tokens"]).to(dev)
    bld["labels"] = torch.from_numpy(bl["labels"]).to(dev)
    bld["emb"], bld["head"] = up(bl["emb"]), up(bl["head"])
    bld["blocks"] = [{k: up(v) for k, v in b.items()} for b in bl["blocks"]]
    # the 12-layer 162M decoder's forward (the byte-LM composition at the
    # model card's shapes): weights resident, buffers and workspaces built once
    dm = inputs.decoder_162m()
    dmd = dict(dm)
    dmd["tokens"] = torch.from_numpy(dm["tokens"]).to(dev)
    dmd["labels"] = torch.from_numpy(dm["labels"]).to(dev)
    dmd["emb"], dmd["head"] = up(dm["emb"]), up(dm["head"])
    dmd["blocks"] = [{k: up(v) for k, v in b.items()} for b in dm["blocks"]]
    dm_blocks = byte_lm.make_blocks(dmd, dev)
    dm_ntok = dm["batch"] * dm["seq"]
    dm_head_ws = detlib.gemm_workspace(dm_ntok, dm["vocab"], dm["d"], False, True, device=dev)
    dm_flops = (len(dm_blocks) * dm_blocks[0].flops()
                + inputs.flops_gemm(dm_ntok, dm["vocab"], dm["d"]))
    # the 162M model's training step at the same size: the forward above, the
    # backward and AdamW on all 162,147,840 parameters; every product of the
    # forward has two of the same size in the backward (dX, dW; for the
    # attention dP, dV and dQ, dK), so 3x the forward's FLOPs (the backward's
    # recomputation of the scores is not counted)
    dm_train_ws = byte_lm.head_workspaces(dmd, dev)
    dm_train_status = torch.zeros(1, dtype=torch.int32, device=dev)
    dm_train_flops = 3 * dm_flops
    digests = input_digests(workload_arrays(fwd, dw, r4, rb, sg, bc, bl, dm, aw))
    # the byte-level LM step is launch-bound (120 small launches): it runs as
    # a CUDA graph captured once, after an eager warm-up that builds its
    # buffers and workspaces
    bl_status = torch.zeros(1, dtype=torch.int32, device=dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        byte_lm.train_step(bld, dev, inputs.BYTE_LM_HP, status=bl_status)
    torch.cuda.current_stream(dev).wait_stream(side)
    bl_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(bl_graph):
        byte_lm.train_step(bld, dev, inputs.BYTE_LM_HP, status=bl_status)
    P, G, Mm, Vv = (up(aw[k]) for k in ("p", "g", "m", "v"))
    hp = {k: aw[k] for k in ("lr", "beta1", "beta2", "eps", "weight_decay", "step")}
    # L2 flush: write 512 MB, then read another 512 MB so the L2 holds clean
    # lines of neither, and no timed kernel pays for the flush's write-backs
    flush = torch.empty(128 * 1024 * 1024, dtype=torch.float32, device=dev)
    flush_r = torch.ones(128 * 1024 * 1024, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    setup_s = time.time() - t_setup

    rows4, D4 = r4["x"].shape
    V = r4["logits"].shape[1]
    n_params = aw["p"].size
    gemm_flops_fwd = [inputs.flops_gemm(*gemm_dims(p)) for p in fwd]
    gemm_flops_dw = [inputs.flops_gemm(*gemm_dims(p)) for p in dw]
    gemm_flops = sum(gemm_flops_fwd) + sum(gemm_flops_dw)
    lm_idx = [p["name"] for p in fwd].index("lm_head")
    # A GEMM is one launch, plus one where it uses its workspace (the split-K
    # second pass, or the transposed copy of A); a group, and the attention,
    # report their own counts. Checked against an ncu launch list of one step.
    def gemm_n(M, N, K, transA=False, transB=False, ws=None):
        # launches of one GEMM with this workspace: the copy of A, the GEMM,
        # the split pass, as its plan takes them
        return detlib.detgemm_launches(M, N, K, transA, transB, ws)

    def planned_n(M, N, K, transA, transB):
        # ... with the workspace its plan asks for
        return gemm_n(M, N, K, transA, transB,
                      detlib.detgemm_workspace_bytes(M, N, K, transA, transB))

    # one block forward: 2 RMSNorms, 5 GEMMs, RoPE, attention, 2 adds, SwiGLU
    attn162 = detlib.detattention_launches(bc["batch"], bc["seq"], inputs.N_HEADS,
                                           bc["x"].shape[1] // inputs.N_HEADS)
    def pair_n(M, N1, N2, K, transA, ws_bytes=None):
        # launches of a two-product group of one shared A (gate/up, or two
        # weight gradients of one input), with the group's own workspace when
        # ws_bytes is None; stand-in tensors carry the shapes
        e = lambda *sh: torch.empty(sh, dtype=torch.float32, device=dev)  # noqa: E731
        A = e(K, M) if transA else e(M, K)
        probs = [dict(A=A, B=e(K, N1), C=e(M, N1), transA=transA),
                 dict(A=A, B=e(K, N2), C=e(M, N2), transA=transA)]
        ws = detlib.gemm_group_workspace(probs) if ws_bytes is None else (
            e(ws_bytes // 4) if ws_bytes else None)
        return detlib.detgemm_group_launches(probs, ws)

    ntok_blk = bc["batch"] * bc["seq"]
    gu_blk = pair_n(ntok_blk, bc["W_gate"].shape[1], bc["W_up"].shape[1],
                    bc["x"].shape[1], False)
    d_blk, f_blk = bc["x"].shape[1], bc["W_gate"].shape[1]
    # a forward block: the first RMSNorm and the fused residual add + second
    # RMSNorm (2), QKV, out, down, the gate/up group, the rotary, the
    # attention, the second residual add and SwiGLU
    block_launches = (2 + gemm_n(ntok_blk, 3 * d_blk, d_blk, ws=blk.ws["qkv"])
                      + gemm_n(ntok_blk, d_blk, d_blk, ws=blk.ws["o"])
                      + gemm_n(ntok_blk, d_blk, f_blk, ws=blk.ws["down"]) + gu_blk
                      + 1 + attn162 + 1 + 1)
    # the byte-level LM step: the embedding, 2 forward blocks (10 launches and
    # the attention), the head GEMM, the cross-entropy and its mean, the head's
    # two backward GEMMs, 2 backward blocks (13 launches, 5 weight-gradient
    # GEMMs and the attention's backward), the embedding backward, and one
    # AdamW launch per parameter tensor (2 + 7 a block); only the
    # weight-gradient GEMMs (K = all tokens) use workspaces
    nb = len(bl["blocks"])
    hd_b = bl["d"] // bl["heads"]
    attn_b = detlib.detattention_launches(bl["batch"], bl["seq"], bl["heads"], hd_b)
    attn_b_bwd = detlib.detattention_launches(bl["batch"], bl["seq"], bl["heads"], hd_b,
                                              backward=True, saved=True)
    ntok_b, d_b, f_b = bl["batch"] * bl["seq"], bl["d"], bl["dff"]

    def dw_n(M, N):
        return planned_n(M, N, ntok_b, True, False)

    def tb_n(M, N, K):
        # an input-gradient GEMM (B transposed) with the workspace its plan asks
        return planned_n(M, N, K, False, True)

    def bwd_block_n(ntok, d, f, attn_bwd, dw):
        # a block's backward: SwiGLU's, the 2 RMSNorm backwards (2 kernels
        # each), 2 adds and the rotary's backward (8); the input gradients
        # through W_down, W_gate, W_up (accumulating), W_o and W_qkv; the
        # weight gradients; the attention's backward
        return (8 + tb_n(ntok, f, d) + 2 * tb_n(ntok, d, f) + tb_n(ntok, d, d)
                + tb_n(ntok, d, 3 * d) + dw + attn_bwd)
    # W_down's, the W_gate/W_up pair's, W_o's and W_qkv's weight gradients
    blk_dw = (dw_n(f_b, d_b) + pair_n(d_b, f_b, f_b, ntok_b, True) + dw_n(d_b, d_b)
              + dw_n(d_b, 3 * d_b))
    # a forward block: the RMSNorm and the fused add + RMSNorm, QKV, out, the
    # gate/up group, down, rotary, the second add, SwiGLU and the attention
    blk_fwd = 2 + 3 + pair_n(ntok_b, f_b, f_b, d_b, False) + 1 + 1 + 1
    # (all blocks but the last leave their second residual add to the next
    # block's first kernel: one launch fewer a block boundary)
    byte_lm_launches = (1 + nb * (blk_fwd + attn_b) - (nb - 1) + 1 + 2
                        + dw_n(bl["vocab"], d_b) + 1
                        + nb * bwd_block_n(ntok_b, d_b, f_b, attn_b_bwd, blk_dw)
                        + 1 + 2 + 7 * nb)
    # the 162M decoder forward: the embedding, 12 blocks as above, the head
    # GEMM (with its transposed copy of the activations), cross-entropy + mean
    decoder_launches = (1 + len(dm_blocks) * block_launches - (len(dm_blocks) - 1)
                        + gemm_n(dm_ntok, dm["vocab"], dm["d"], False, True, dm_head_ws) + 2)
    # its training step: that forward; the head's dW and dX GEMMs; each
    # block's backward (as above, with its workspaces); the embedding backward;
    # AdamW per parameter tensor
    nb_m, d_m, f_m = len(dm_blocks), dm["d"], dm["dff"]

    def dw_m(M, N):
        return planned_n(M, N, dm_ntok, True, False)
    attn_m_bwd = detlib.detattention_launches(dm["batch"], dm["seq"], dm["heads"],
                                              d_m // dm["heads"], backward=True, saved=True)
    blk_dw_m = (dw_m(f_m, d_m) + pair_n(d_m, f_m, f_m, dm_ntok, True) + dw_m(d_m, d_m)
                + dw_m(d_m, 3 * d_m))
    train_launches = (decoder_launches
                      + gemm_n(dm["vocab"], d_m, dm_ntok, True, False, dm_train_ws["head_dw"])
                      + gemm_n(dm_ntok, d_m, dm["vocab"], False, False, dm_train_ws["head_dx"])
                      + nb_m * bwd_block_n(dm_ntok, d_m, f_m, attn_m_bwd, blk_dw_m)
                      + 1 + 2 + 7 * nb_m)
    dw_launches = detlib.detgemm_group_launches(dw_probs, ws_dw)
    fwd_launches = (sum(gemm_n(*gemm_dims(p), p["transA"], p["transB"], ws_fwd[i])
                        for i, p in enumerate(fwd) if i not in gu)
                    + detlib.detgemm_group_launches(gu_probs, ws_gu))
    launches_per_step = (1 + RMS_RUN + fwd_launches + 2 + 2 * (1 + RMSB_RUN)
                         + dw_launches + 1 + block_launches
                         + byte_lm_launches + decoder_launches + train_launches + 1)

    segs = ["rmsnorm_1", "rmsnorm", "gemm_fwd_other", "gemm_lm_head", "xent", "rmsnorm_bwd_1",
            "rmsnorm_bwd", "gemm_dw", "shard_sum", "block_fwd", "byte_lm_step", "forward_162m",
            "train_162m", "adamw"]

    def step(ev=None):
        marks = iter(range(len(segs) + 1))

        def mark():
            i = next(marks)
            if ev is not None:
                ev[i].record()
        mark()
        detlib.detrmsnorm_f32(x4, gain4, float(r4["eps"]), y=y4, inv_rms=inv4)
        mark()
        for xr, yr, ir in rms_runs:
            detlib.detrmsnorm_f32(xr, gain4, float(r4["eps"]), y=yr, inv_rms=ir)
        mark()
        for i, (p, A, B) in enumerate(g_fwd):
            if i == lm_idx or i == gu[1]:
                continue
            if i == gu[0]:
                detlib.detgemm_group_f32(gu_probs, workspace=ws_gu)
                continue
            detlib.detgemm_f32(A, B, c_fwd[i], transA=p["transA"], transB=p["transB"],
                               workspace=ws_fwd[i])
        mark()
        p, A, B = g_fwd[lm_idx]
        detlib.detgemm_f32(A, B, c_fwd[lm_idx], transA=p["transA"], transB=p["transB"],
                           workspace=ws_fwd[lm_idx])
        mark()
        detlib.detxent_f32(logits, labels, loss=loss, loss_mean=lmean, dlogits=dlog,
                           dscale=1.0 / rows4, dev_status=status)
        mark()
        detlib.detrmsnorm_bwd_f32(x4, gain4, inv4, dy4, dx=dx4, dgain=dgain4, workspace=ws_rb)
        mark()
        for xr, dyr, dxr, dgr in rmsb_runs:
            detlib.detrmsnorm_bwd_f32(xr, gain4, inv4, dyr, dx=dxr, dgain=dgr, workspace=ws_rb)
        mark()
        detlib.detgemm_group_f32(dw_probs, workspace=ws_dw)
        mark()
        detlib.detshardsum_f32(shards, scale=1.0 / shards.shape[0], out=gsum)
        mark()
        blk.forward(bx, bw)
        mark()
        bl_graph.replay()
        mark()
        byte_lm.forward(dmd, dev, blocks=dm_blocks, head_ws=dm_head_ws)
        mark()
        byte_lm.train_step(dmd, dev, inputs.BYTE_LM_HP, status=dm_train_status,
                           blocks=dm_blocks, ws=dm_train_ws)
        mark()
        detlib.detadamw_f32(P, G, Mm, Vv, **hp)
        mark()

    import torch.distributed as dist
    distributed = world > 1

    def barrier():
        if distributed:
            dist.barrier()
        torch.cuda.synchronize()

    def flush_l2(v):
        flush.fill_(v)
        return flush_r.sum()

    for _ in range(args.warmup):
        flush_l2(1.0)
        step()
    barrier()

    sampler = ClockSampler(local_rank)
    sampler.start()
    events = []
    barrier()
    t0 = time.time()
    for _ in range(args.steps):
        flush_l2(float(len(events)))             # L2 flush, outside the events
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(segs) + 1)]
        step(ev)
        events.append(ev)
    barrier()
    wall = time.time() - t0
    clocks = sampler.stop()

    seg_ms = {s: 0.0 for s in segs}
    for ev in events:
        for i, s in enumerate(segs):
            seg_ms[s] += ev[i].elapsed_time(ev[i + 1])
    step_ms = sum(seg_ms.values()) / args.steps
    gemm_ms = (seg_ms["gemm_fwd_other"] + seg_ms["gemm_lm_head"] + seg_ms["gemm_dw"]) / args.steps
    lm_ms = seg_ms["gemm_lm_head"] / args.steps

    # max over ranks of the per-step device times
    if distributed:
        vals = max_over_ranks([step_ms, gemm_ms, lm_ms] + [seg_ms[s] for s in segs], dev)
        step_ms, gemm_ms, lm_ms = vals[:3]
        for i, s in enumerate(segs):
            seg_ms[s] = vals[3 + i]

    if int(status.item()) != 0:
        raise SystemExit("cross-entropy reported an out-of-range label")
    if int(bl_status.item()) != 0:
        raise SystemExit("the byte-LM step reported an out-of-range token or label")
    if int(dm_train_status.item()) != 0:
        raise SystemExit("the 162M training step reported an out-of-range token or label")
    if detlib.det_watchdog_status() != 0:
        raise SystemExit("a bounded device wait gave up during the run")

    result = None
    if rank == 0:
        peaks, peak_kind = measured_peaks()
        hbm = float(peaks["hbm_gbs"])
        smax = float(peaks.get("sm_max_mhz", 2070.0))
        fma_peak = fp32_peak_tflops(smax)
        per = lambda s: seg_ms[s] / args.steps / 1e3   # seconds a step
        gemm_tflops = replica_throughput(gemm_flops, world, gemm_ms) / 1e12
        lm_flops = gemm_flops_fwd[lm_idx]
        lm_tflops = lm_flops / (lm_ms / 1e3) / 1e12
        ops = {
            "gemm_all": {"tflops": gemm_tflops / world, "frac_fp32_peak": gemm_tflops / world / fma_peak,
                         "ms": gemm_ms},
            "gemm_lm_head": {"tflops": lm_tflops, "frac_fp32_peak": lm_tflops / fma_peak,
                             "ms": lm_ms},
            "gemm_fwd_other": {"tflops": (sum(gemm_flops_fwd) - lm_flops) / per("gemm_fwd_other") / 1e12,
                               "ms": per("gemm_fwd_other") * 1e3},
            "gemm_dw": {"tflops": sum(gemm_flops_dw) / per("gemm_dw") / 1e12,
                        "ms": per("gemm_dw") * 1e3},
            "rmsnorm": hbm_row(bytes_rmsnorm(rows4, D4), per("rmsnorm") / RMS_RUN, hbm,
                               launches=RMS_RUN,
                               one_launch=hbm_row(bytes_rmsnorm(rows4, D4), per("rmsnorm_1"), hbm)),
            "rmsnorm_bwd": hbm_row(bytes_rmsnorm_bwd(rows4, D4), per("rmsnorm_bwd") / RMSB_RUN, hbm,
                                   launches=RMSB_RUN,
                                   one_launch=hbm_row(bytes_rmsnorm_bwd(rows4, D4),
                                                      per("rmsnorm_bwd_1"), hbm)),
            "block_fwd": {"tflops": blk.flops() / per("block_fwd") / 1e12,
                          "frac_fp32_peak": blk.flops() / per("block_fwd") / 1e12 / fma_peak,
                          "ms": per("block_fwd") * 1e3},
            "byte_lm_step": {"ms": per("byte_lm_step") * 1e3,
                             "tokens_per_s": bl["batch"] * bl["seq"] / per("byte_lm_step")},
            "forward_162m": {"ms": per("forward_162m") * 1e3,
                             "tokens_per_s": dm_ntok / per("forward_162m"),
                             "tflops": dm_flops / per("forward_162m") / 1e12,
                             "frac_fp32_peak": dm_flops / per("forward_162m") / 1e12 / fma_peak},
            "train_162m": {"ms": per("train_162m") * 1e3,
                           "tokens_per_s": dm_ntok / per("train_162m"),
                           "tflops": dm_train_flops / per("train_162m") / 1e12,
                           "frac_fp32_peak": dm_train_flops / per("train_162m") / 1e12 / fma_peak},
            "shard_sum": {"gbs": bytes_shardsum(*sg.shape) / per("shard_sum") / 1e9,
                          "frac_hbm": bytes_shardsum(*sg.shape) / per("shard_sum") / 1e9 / hbm,
                          "ms": per("shard_sum") * 1e3},
            "xent": {"gbs": bytes_xent(rows4, V) / per("xent") / 1e9,
                     "frac_hbm": bytes_xent(rows4, V) / per("xent") / 1e9 / hbm,
                     "ms": per("xent") * 1e3},
            "adamw": {"gbs": bytes_adamw(n_params) / per("adamw") / 1e9,
                      "frac_hbm": bytes_adamw(n_params) / per("adamw") / 1e9 / hbm,
                      "ms": per("adamw") * 1e3},
        }
        traffic = load_traffic()
        result = {
            "metric": METRIC,
            "value": round(gemm_tflops, 4),
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(step_ms, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic (seeded numpy PCG64, shapes of the 162M model card)",
            "input_sha256": digests,
            "config": {"workload": WORKLOAD, "tokens": rows4, "d_model": D4, "vocab": V,
                       "params": int(n_params), "parallelism": f"replicas{world}",
                       "l2": "flushed before every timed step (512 MB write, then 512 MB read "
                                     "of another buffer)"},
            "roofline": {"bound": "alu", "kernel": "gemm_kernel (LM head, 8192x50257x768)",
                         "achieved": round(lm_tflops, 4),
                         "peak": round(fma_peak, 3), "unit": "TFLOP/s",
                         "frac": round(lm_tflops / fma_peak, 4),
                         "peak_kind": f"FP32 FFMA: {SM_COUNT} SMs x 128 lanes x 2 x "
                                      f"{smax:.0f} MHz ({peak_kind} max clock)",
                         "traffic": traffic.get("gemm_lm_head")},
            "rooflines": {
                "rmsnorm": {"bound": "hbm", "achieved": round(ops["rmsnorm"]["gbs"], 1),
                            "peak": hbm, "unit": "GB/s",
                            "frac": round(ops["rmsnorm"]["frac_hbm"], 4),
                            "traffic": traffic.get("rmsnorm"),
                            "timing": f"mean of {RMS_RUN} back-to-back launches over distinct "
                                      "inputs; one launch alone: "
                                      f"{ops['rmsnorm']['one_launch']['frac_hbm']:.4f}"},
                "rmsnorm_bwd": {"bound": "hbm", "achieved": round(ops["rmsnorm_bwd"]["gbs"], 1),
                                "peak": hbm, "unit": "GB/s",
                                "frac": round(ops["rmsnorm_bwd"]["frac_hbm"], 4),
                                "traffic": traffic.get("rmsnorm_bwd"),
                                "timing": f"mean of {RMSB_RUN} back-to-back launches over "
                                          "distinct inputs; one launch alone: "
                                          f"{ops['rmsnorm_bwd']['one_launch']['frac_hbm']:.4f}"},
                "shard_sum": {"bound": "hbm", "achieved": round(ops["shard_sum"]["gbs"], 1),
                              "peak": hbm, "unit": "GB/s",
                              "frac": round(ops["shard_sum"]["frac_hbm"], 4),
                              "traffic": traffic.get("shard_sum")},
                "xent": {"bound": "hbm", "achieved": round(ops["xent"]["gbs"], 1),
                         "peak": hbm, "unit": "GB/s",
                         "frac": round(ops["xent"]["frac_hbm"], 4),
                         "traffic": traffic.get("xent")},
                "adamw": {"bound": "hbm", "achieved": round(ops["adamw"]["gbs"], 1),
                          "peak": hbm, "unit": "GB/s",
                          "frac": round(ops["adamw"]["frac_hbm"], 4),
                          "traffic": traffic.get("adamw")},
                "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"},
            "ops": ops,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "setup_s": round(setup_s, 1),
            "timed_wall_s": round(wall, 3),
        }
        if not args.skip_e2e:
            result["e2e"] = e2e_leg(args, dev, host, gemm_flops)
        if not args.skip_cpu and world == 1:
            result["cpu_baseline"] = cpu_baseline(args)
    return result


def load_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, when present and
    current (profiles/traffic.json; null otherwise)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return {}
    try:
        return {k: v for k, v in json.load(open(path)).get("per_launch_bytes", {}).items()}
    except (OSError, ValueError):
        return {}


def e2e_leg(args, dev, host, gemm_flops):
    """The same step through the public API with pinned host buffers: every
    input copied host->device and every output device->host inside the timed
    region, each step. Copies in, compute and copies out run on three streams,
    so one op's outputs drain while later ops' inputs arrive and run."""
    import torch

    from bitwise_reproducible_fp32_gb300 import detlib

    fwd, dw, r4, rb, sg, aw = (host[k] for k in ("fwd", "dw", "r4", "rb", "sg", "aw"))
    pinned = {}

    def pin(a):
        k = id(a)
        if k not in pinned:
            t = torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
            pinned[k] = (t, torch.empty(t.shape, dtype=t.dtype, device=dev))
        return pinned[k]

    srcs = []
    for p in fwd + dw:
        srcs += [pin(p["A"]), pin(p["B"])]
    for k in ("x", "gain", "logits", "labels"):
        srcs.append(pin(r4[k]))
    srcs.append(pin(rb["dy"]))
    srcs.append(pin(sg))
    for k in ("p", "g", "m", "v"):
        srcs.append(pin(aw[k]))
    uniq = list({id(s[0]): s for s in srcs}.values())
    h2d = sum(t.numel() * t.element_size() for t, _ in uniq)

    outs_dev = [torch.empty(gemm_dims(p)[:2], dtype=torch.float32, device=dev)
                for p in fwd + dw]
    wss = [detlib.gemm_workspace(*gemm_dims(p), p["transA"], p["transB"], device=dev)
           for p in fwd]
    rows4, D4 = r4["x"].shape
    V = r4["logits"].shape[1]
    y4 = torch.empty((rows4, D4), dtype=torch.float32, device=dev)
    inv4 = torch.empty(rows4, dtype=torch.float32, device=dev)
    loss = torch.empty(rows4, dtype=torch.float32, device=dev)
    lmean = torch.empty(1, dtype=torch.float32, device=dev)
    dlog = torch.empty((rows4, V), dtype=torch.float32, device=dev)
    dx4 = torch.empty((rows4, D4), dtype=torch.float32, device=dev)
    dgain4 = torch.empty(D4, dtype=torch.float32, device=dev)
    ws_rb = torch.empty((detlib.detrmsnorm_bwd_workspace_bytes(rows4, D4) + 3) // 4,
                        dtype=torch.float32, device=dev)
    gsum = torch.empty(sg.shape[1], dtype=torch.float32, device=dev)
    dev_outs = outs_dev + [y4, inv4, loss, lmean, dlog, dx4, dgain4, gsum]
    host_outs = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dev_outs]
    pmv_host = [torch.empty(aw[k].shape, dtype=torch.float32).pin_memory()
                for k in ("p", "m", "v")]
    d2h = sum(t.numel() * 4 for t in host_outs) + sum(t.numel() * 4 for t in pmv_host)
    hp = {k: aw[k] for k in ("lr", "beta1", "beta2", "eps", "weight_decay", "step")}

    g = lambda a: pin(a)[1]                                    # noqa: E731
    P, G, M, Vv = (g(aw[k]) for k in ("p", "g", "m", "v"))
    # (inputs, call, outputs) in step order: each op's inputs are copied in on
    # one stream, the op runs on the compute stream once they have landed, and
    # its outputs are copied out on a third stream while later ops run. The
    # host link carries 5.2 GB in and 5.6 GB out, so the order keeps the
    # device-to-host stream busy from early on: the LM head first, in row
    # blocks whose outputs drain while the next blocks run; AdamW in element
    # blocks that run as their state arrives. A row block of a GEMM, and an
    # element block of AdamW, compute exactly the bits of the whole call.
    ops = []
    names = [p["name"] for p in fwd]
    gu = (names.index("swiglu_gate"), names.index("swiglu_up"))
    lm = names.index("lm_head")
    nf = len(fwd)
    dwp = [dict(A=g(p["A"]), B=g(p["B"]), C=outs_dev[nf + j], transA=p["transA"],
                transB=p["transB"]) for j, p in enumerate(dw)]
    ws_dwp = detlib.gemm_group_workspace(dwp, device=dev)
    ops_dw = ([t for p in dw for t in (pin(p["A"]), pin(p["B"]))],
              lambda: detlib.detgemm_group_f32(dwp, workspace=ws_dwp),
              [(outs_dev[nf + j], host_outs[nf + j]) for j in range(len(dw))])
    # the LM head by row blocks of E2E_LM_ROWS tokens (one workspace, reused in
    # stream order)
    p_lm = fwd[lm]
    A_lm, B_lm, C_lm, hC_lm = g(p_lm["A"]), g(p_lm["B"]), outs_dev[lm], host_outs[lm]
    rows_lm = A_lm.shape[0]
    blk = min(E2E_LM_ROWS, rows_lm)
    ws_lm = detlib.gemm_workspace(blk, *gemm_dims(p_lm)[1:], p_lm["transA"], p_lm["transB"],
                                  device=dev)
    for r0 in range(0, rows_lm, blk):
        r1 = min(rows_lm, r0 + blk)
        ops.append(([pin(p_lm["A"]), pin(p_lm["B"])] if r0 == 0 else [],
                    lambda r0=r0, r1=r1: detlib.detgemm_f32(
                        A_lm[r0:r1], B_lm, C_lm[r0:r1], transA=p_lm["transA"],
                        transB=p_lm["transB"], workspace=ws_lm),
                    [(C_lm[r0:r1], hC_lm[r0:r1])]))
    for i, p in enumerate(fwd):
        if i == gu[1] or i == lm:
            continue
        if i == gu[0]:
            # the gate and up projections as one group, as in the device-timed step
            q0, q1 = fwd[gu[0]], fwd[gu[1]]
            gu_probs = [dict(A=g(q0["A"]), B=g(q0["B"]), C=outs_dev[gu[0]]),
                        dict(A=g(q1["A"]), B=g(q1["B"]), C=outs_dev[gu[1]])]
            ws_gu = detlib.gemm_group_workspace(gu_probs, device=dev)
            ops.append(([pin(q0["A"]), pin(q0["B"]), pin(q1["B"])],
                        lambda gp=gu_probs, w=ws_gu: detlib.detgemm_group_f32(gp, workspace=w),
                        [(outs_dev[j], host_outs[j]) for j in gu]))
            continue
        ops.append(([pin(p["A"]), pin(p["B"])],
                    lambda i=i, p=p: detlib.detgemm_f32(g(p["A"]), g(p["B"]), outs_dev[i],
                                                        transA=p["transA"], transB=p["transB"],
                                                        workspace=wss[i]),
                    [(outs_dev[i], host_outs[i])]))
    n = len(fwd + dw)
    ops.append(([pin(r4["x"]), pin(r4["gain"])],
                lambda: detlib.detrmsnorm_f32(g(r4["x"]), g(r4["gain"]), float(r4["eps"]), y=y4,
                                              inv_rms=inv4),
                [(y4, host_outs[n]), (inv4, host_outs[n + 1])]))
    ops.append(([pin(r4["logits"]), pin(r4["labels"])],
                lambda: detlib.detxent_f32(g(r4["logits"]), g(r4["labels"]), loss=loss,
                                           loss_mean=lmean, dlogits=dlog, dscale=1.0 / rows4),
                [(loss, host_outs[n + 2]), (lmean, host_outs[n + 3]), (dlog, host_outs[n + 4])]))
    # AdamW by element blocks: each block's p, g, m, v are copied in as views of
    # the pinned host arrays, and its p, m, v copied out
    n_p = P.numel()
    eb = (n_p + E2E_ADAMW_BLOCKS - 1) // E2E_ADAMW_BLOCKS
    eb = (eb + 255) // 256 * 256
    host_pgmv = [pin(aw[k])[0] for k in ("p", "g", "m", "v")]
    for e0 in range(0, n_p, eb):
        e1 = min(n_p, e0 + eb)
        ins = [(h[e0:e1], d[e0:e1]) for h, d in zip(host_pgmv, (P, G, M, Vv))]
        ops.append((ins,
                    lambda e0=e0, e1=e1: detlib.detadamw_f32(P[e0:e1], G[e0:e1], M[e0:e1],
                                                             Vv[e0:e1], **hp),
                    [(d[e0:e1], h[e0:e1]) for d, h in zip((P, M, Vv), pmv_host)]))
    ops.append(([pin(rb["dy"])],
                lambda: detlib.detrmsnorm_bwd_f32(g(r4["x"]), g(r4["gain"]), inv4, g(rb["dy"]),
                                                  dx=dx4, dgain=dgain4, workspace=ws_rb),
                [(dx4, host_outs[n + 5]), (dgain4, host_outs[n + 6])]))
    ops.append(ops_dw)          # the weight-gradient GEMMs as one group
    ops.append(([pin(sg)], lambda: detlib.detshardsum_f32(g(sg), scale=1.0 / sg.shape[0], out=gsum),
                [(gsum, host_outs[n + 7])]))
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def one_step():
        s_in.wait_stream(comp)      # the previous step is done with the inputs
        landed, seen = [], set()
        with torch.cuda.stream(s_in):
            for inputs, _, _ in ops:
                for t, d in inputs:
                    if id(t) not in seen:
                        d.copy_(t, non_blocking=True)
                        seen.add(id(t))
                ev = torch.cuda.Event()
                ev.record(s_in)
                landed.append(ev)
        for (_, call, outs), ev in zip(ops, landed):
            comp.wait_event(ev)
            call()
            done = torch.cuda.Event()
            done.record(comp)
            s_out.wait_event(done)
            with torch.cuda.stream(s_out):
                for d, h in outs:
                    h.copy_(d, non_blocking=True)
        comp.wait_stream(s_out)     # the step ends with its outputs on the host

    for _ in range(max(1, min(args.warmup, 3))):
        one_step()
    torch.cuda.synchronize()
    # each step timed on its own (host wall clock, synchronised on both sides);
    # the median of the steps is reported, as a step's host copies vary with
    # what else the host link carries
    steps = max(1, min(args.steps, 7))
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        one_step()
        torch.cuda.synchronize()
        times.append(time.perf_counter() - t0)
    dt = sorted(times)[len(times) // 2]
    return {"value": round(gemm_flops / dt / 1e12, 4), "unit": "TFLOP/s",
            "ms_per_step": round(dt * 1e3, 3), "steps": steps,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


# ------------------------------------------------------------------ oracle legs
def oracle_sample(budget_s: float):
    """Times the CPU oracle on bounded samples of the step's operations, on all
    host cores. Returns the rates and a description."""
    import oracle

    oracle.build()
    cores = oracle.nthreads_default()
    fwd, _ = gemm_list()
    lm = [p for p in fwd if p["name"] == "lm_head"][0]
    rates = {}
    # GEMM: rows of the LM head until the time budget is spent
    rows_done, t_g, flops = 0, 0.0, 0
    step_rows = max(cores, 16)
    while t_g < budget_s * 0.6 and rows_done + step_rows <= lm["A"].shape[0]:
        a = np.ascontiguousarray(lm["A"][rows_done:rows_done + step_rows])
        t0 = time.perf_counter()
        oracle.gemm(a, lm["B"], transB=True, nthreads=cores)
        t_g += time.perf_counter() - t0
        rows_done += step_rows
        flops += 2 * step_rows * lm["B"].shape[0] * lm["B"].shape[1]
    rates["gemm_tflops"] = flops / t_g / 1e12
    r4 = inputs.rowops_cfg4(rows=cores * 4)
    t0 = time.perf_counter()
    oracle.xent(r4["logits"], r4["labels"], with_dlogits=True, nthreads=cores)
    dt = time.perf_counter() - t0
    rates["xent_gbs"] = bytes_xent(*r4["logits"].shape) / dt / 1e9
    t0 = time.perf_counter()
    oracle.rmsnorm(r4["x"], r4["gain"], eps=r4["eps"], nthreads=cores)
    dt = time.perf_counter() - t0
    rates["rmsnorm_gbs"] = bytes_rmsnorm(*r4["x"].shape) / dt / 1e9
    rb = inputs.rmsnorm_bwd_cfg4(rows=512)          # two 256-row chunks
    _, inv = oracle.rmsnorm(rb["x"], rb["gain"], eps=rb["eps"], nthreads=cores)
    t0 = time.perf_counter()
    oracle.rmsnorm_bwd(rb["x"], rb["gain"], inv, rb["dy"], nthreads=cores)
    dt = time.perf_counter() - t0
    rates["rmsnorm_bwd_gbs"] = bytes_rmsnorm_bwd(*rb["x"].shape) / dt / 1e9
    sg = inputs.shard_grads(n=200_000)
    t0 = time.perf_counter()
    oracle.shardsum(sg, scale=1.0 / sg.shape[0], nthreads=cores)
    dt = time.perf_counter() - t0
    rates["shard_sum_gbs"] = bytes_shardsum(*sg.shape) / dt / 1e9
    n = 20_000_000
    a = inputs.adamw_cfg5(n=n)
    t0 = time.perf_counter()
    oracle.adamw(a["p"], a["g"], a["m"], a["v"], a["lr"], a["beta1"], a["beta2"],
                 a["eps"], a["weight_decay"], a["step"], nthreads=cores)
    dt = time.perf_counter() - t0
    rates["adamw_gbs"] = bytes_adamw(n) / dt / 1e9
    sample = (f"LM-head GEMM rows 0..{rows_done - 1} of 8192 (x 50257 x 768, "
              f"{flops / 1e9:.1f} GFLOP); xent {r4['logits'].shape[0]} rows x 50257 "
              f"with dlogits; RMSNorm {r4['x'].shape[0]} rows; RMSNorm backward 512 rows; "
              f"shard sum 64 x 200000; AdamW {n} params")
    return rates, cores, sample


def cpu_baseline(args):
    rates, cores, sample = oracle_sample(budget_s=args.cpu_budget)
    return {"value": round(rates["gemm_tflops"], 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle", "sample": sample,
            "ops": {k: round(v, 4) for k, v in rates.items()}}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, on a bounded sample of
    the workload each step."""
    if rank != 0:
        return None
    for _ in range(args.warmup):
        oracle_sample(budget_s=0.5)
    vals, last = [], None
    t0 = time.perf_counter()
    for _ in range(args.steps):
        last = oracle_sample(budget_s=max(1.0, args.cpu_budget / max(args.steps, 1)))
        vals.append(last[0]["gemm_tflops"])
    wall = time.perf_counter() - t0
    value = statistics.median(vals)
    rates, cores, sample = last
    return {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "impl": "reference", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(wall / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded numpy PCG64)",
            "config": {"workload": WORKLOAD, "parallelism": f"replicas{world}",
                       "sample_per_step": sample},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "kind": "oracle",
                             "cores": cores, "sample": sample,
                             "ops": {k: round(v, 4) for k, v in rates.items()}},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle GEMM work in the CPU baseline")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
