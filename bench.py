"""Benchmark of the multi-LoRA decode hot path on GB300.

One step = one pass of the whole path over the decode batches of the
Llama-3-8B q/k/v workload (H=4096, q/k/v slices 4096/1024/1024, rank 16,
4 adapters, bf16, 10 % of tokens without an adapter; one batch each of
T = 16, 128, 256, 512, 1024 tokens): for every batch, BGMV grouping of the
token indices, the stacked q/k/v shrink into the fp32 rank buffer, and the
three-slice expand_slice into the fused q/k/v output (add_inputs, as vLLM
PR #11579 benchmarks the expand).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores on the same workload instead (bounded samples per step).
Multi-GPU (torchrun): every rank runs its own batches, no collective on the
data path (weak scaling); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from typing import Optional

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import lora_inputs as li  # noqa: E402

METRIC = "LoRA shrink+expand tokens/s and achieved % of HBM/tensor roofline (1×GB300)"
WORKLOAD = ("decode BGMV, Llama-3-8B q/k/v: H=4096, expand_slice into q/k/v slices "
            "4096/1024/1024, r=16, L=4 adapters, bf16, T in {16,128,256,512,1024} "
            "(one batch of each per step), idx uniform over adapters, 10% idx=-1, "
            "weights N(0,0.02), add_inputs=True")
H, R, L, SLICES = 4096, 16, 4, li.QKV_SLICES
NTOT = sum(SLICES)
E = 2  # bytes per bf16 element
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(ms_local: float, tokens_local: int, ws: int, device=None):
    """Whole-job figures over ranks that run independent batches (replicas,
    no data-path collective): the slowest rank's time and every rank's
    tokens.  Returns (ms, tokens, tokens_per_s)."""
    ms, tokens = float(ms_local), float(tokens_local)
    if ws > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        n = torch.tensor([tokens], dtype=torch.float64, device=device)
        dist.all_reduce(n, op=dist.ReduceOp.SUM)
        ms, tokens = float(t.item()), float(n.item())
    return ms, tokens, tokens / (ms / 1e3)


# ---------------------------------------------------------------- work model

def algorithmic(idx: torch.Tensor):
    """Algorithmic bytes / flops of one batch (what the method must move).

    shrink: x rows of active tokens + live A rows of used adapters + y written
    expand_slice: y rows read + live B rows of used adapters + out read and
                  written for active tokens (add_inputs)."""
    T = idx.numel()
    act = idx >= 0
    Ta = int(act.sum())
    U = int(torch.unique(idx[act]).numel())
    S = len(SLICES)
    sh_bytes = Ta * H * E + U * S * R * H * E + T * S * R * 4
    sh_flops = 2 * H * S * R * Ta
    ex_bytes = Ta * S * R * 4 + U * NTOT * R * E + 2 * Ta * NTOT * E
    ex_flops = 2 * NTOT * R * Ta
    return sh_bytes, sh_flops, ex_bytes, ex_flops


def segment_work(T: int, Hm: int, N: int, r: int, S: int, U: int):
    """Algorithmic bytes / flops of an SGMV batch in which every token is
    active (fp16/bf16 operands, fp32 y, add_inputs=True): shrink = x + live
    A rows + y written; expand_slice = y read + live B rows + out read and
    written, over S slices of N columns each."""
    sh_b = T * Hm * E + U * S * r * Hm * E + T * S * r * 4
    sh_f = 2 * T * Hm * S * r
    ex_b = T * S * r * 4 + U * S * N * r * E + 2 * T * S * N * E
    ex_f = 2 * T * S * N * r
    return sh_b, sh_f, ex_b, ex_f


def single_slice_work(Ta: int, T: int, U: int, Hm: int, N: int, r: int, add: bool):
    """Algorithmic bytes of one shrink and one single-slice expand: shrink =
    x rows of the Ta active tokens + live A rows of the U used adapters + y
    written for all T tokens; expand = y rows read + live B rows + out read
    and written (add_inputs) or written for every token (without)."""
    sh_b = Ta * Hm * E + U * r * Hm * E + T * r * 4
    ex_b = Ta * r * 4 + U * N * r * E + (2 * Ta * N * E if add else T * N * E)
    return sh_b, ex_b


def prefill_sgmv(lg, dev, hbm_gbs: float, tc_tflops: float, reps: int = 20):
    """The prefill SGMV gate/up workload (8 segments, log-uniform lengths in
    [8, 2048], adapters A A A B C C D D, H = 4096, gate/up slices of 14336,
    fp16), per rank r: shrink and expand_slice each timed with CUDA events
    around a graph of `reps` back-to-back launches (x rotated over copies
    larger than L2, out > L2), against the roofline max(algorithmic bytes /
    HBM, flops / tensor peak)."""
    res = {}
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    for r in (16, 32, 64):
        c = li.prefill_gateup(r=r)
        T, S, N = c.T, c.num_slices, c.B[0].shape[1]
        U = int(torch.unique(c.seg_lora[c.seg_len > 0]).numel())
        ncopy = max(2, -(-2 * l2 // (T * H * 2)))
        xs = [c.x.to(dev) for _ in range(ncopy)]
        ys = [torch.empty(T, S * r, dtype=torch.float32, device=dev) for _ in range(ncopy)]
        A = c.A.to(dev)
        Bs = [b.to(dev) for b in c.B]
        out = c.out.to(dev)
        plan = lg.new_plan(T, c.L, dev)
        lg.lora_group_segments(c.seg_start.to(dev), c.seg_len.to(dev), c.seg_lora.to(dev), T, c.L,
                               plan)
        torch.cuda.synchronize()

        def timed(launch):
            stream = torch.cuda.Stream()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(reps):
                    launch(i % ncopy)
            g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / reps / 1e3

        t_sh = timed(lambda i: lg.lora_shrink(xs[i], A, ys[i], plan, num_slices=S))
        t_ex = timed(lambda i: lg.lora_expand_slice(ys[i], Bs, out, plan, c.slice_offsets,
                                                    y_slice_stride=r, add_inputs=True))
        sh_b, sh_f, ex_b, ex_f = segment_work(T, H, N, r, S, U)
        out_r = {"T": T}
        for name, t, b, f in (("shrink", t_sh, sh_b, sh_f), ("expand_slice", t_ex, ex_b, ex_f)):
            t_mem, t_tc = b / (hbm_gbs * 1e9), f / (tc_tflops * 1e12)
            out_r[name] = {"us": t * 1e6, "GBps": b / t / 1e9, "TFLOPs": f / t / 1e12,
                           "bound": "hbm" if t_mem >= t_tc else "tensor",
                           "roofline_frac": max(t_mem, t_tc) / t}
        res[f"r{r}"] = out_r
        del xs, ys, out
    return res


def pool_op_us(make_set, launch, set_bytes: int, l2_bytes: int, reps: int = 5,
               max_sets: int = 512):
    """Average duration of one operator launch: `make_set(i)` builds argument
    set i on the device; enough sets that together they are >= 4x L2 (so each
    launch reads from HBM), one launch per set captured in a CUDA graph,
    replayed `reps` times between two events on the launching stream."""
    nsets = int(min(max_sets, max(2, -(-4 * l2_bytes // max(set_bytes, 1)))))
    sets = [make_set(i) for i in range(nsets)]
    launch(sets[0])  # first use outside the capture (library handles, lazy setup)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for a in sets:
            launch(a)
    g.replay()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(reps):
        g.replay()
    t1.record()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) * 1e3 / (reps * nsets), nsets


def next_rows(lg, dev, hbm_gbs: float):
    """The widening rows after the decode and prefill paths:
    - the microbenchmark PR's printed point (SGMV expand, m = 256 as 16
      requests x 16 tokens, r = 16, n = 2048, 4 adapters sorted by id,
      add_inputs=False) beside torch.mm of the same shape (f16 [256,16] x
      [16,2048]), the pages' own two figures given for context;
    - the single-adapter dense case of that shape (one segment, one adapter)
      against the same torch.mm;
    - Llama-3 o_proj / down_proj shapes at decode batches T = 16 and 1024
      (BGMV, r = 16, 4 adapters, 10 % idx = -1, bf16), shrink and expand.
    Each figure is the average launch over a rotating pool of argument sets
    >= 4x L2, against the HBM roofline (algorithmic bytes / measured copy
    bandwidth)."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    res = {}

    def point(c, tag):
        T, N, r = c.T, c.B[0].shape[1], c.R
        U = int(torch.unique(c.seg_lora[c.seg_len > 0]).numel())
        plan = lg.new_plan(T, c.L, dev)
        lg.lora_group_segments(c.seg_start.to(dev), c.seg_len.to(dev), c.seg_lora.to(dev), T,
                               c.L, plan)
        B0, out0 = c.B[0].to(dev), c.out.to(dev)
        g = torch.Generator(device="cpu").manual_seed(3)
        y0 = torch.randn(T, r, generator=g).to(dev)
        _, ex_bytes = single_slice_work(T, T, U, c.A.shape[2], N, r, add=False)
        sb = ex_bytes

        def mk(i):
            return {"y": y0.clone(), "B": B0.clone(), "out": out0.clone()}

        t_ex, n = pool_op_us(mk, lambda a: lg.lora_expand(a["y"], a["B"], a["out"], plan,
                                                          add_inputs=False), sb, l2)
        # the plan-free operator on the same batch: per-token indices, or none
        # at all when one adapter serves every token (the mask-free case)
        single = U == 1 and int(c.seg_lora[0]) == 0 and int(c.seg_len.sum()) == T
        idx_d = None if single else c.lora_of_token().to(dev)
        t_bg, _ = pool_op_us(mk, lambda a: lg.lora_bgmv_expand_slice(
            a["y"], [a["B"]], a["out"], [0], idx_d, y_slice_stride=0, add_inputs=False), sb, l2)
        a16 = y0.to(torch.float16)
        b16 = B0[0].t().contiguous()

        def mk_mm(i):
            return {"a": a16.clone(), "b": b16.clone(), "c": torch.empty(T, N, dtype=torch.float16,
                                                                         device=dev)}

        mm_bytes = T * r * 2 + r * N * 2 + T * N * 2
        t_mm, _ = pool_op_us(mk_mm, lambda a: torch.mm(a["a"], a["b"], out=a["c"]), mm_bytes, l2)
        return {"workload": tag, "expand_us": t_ex, "expand_GBps": ex_bytes / t_ex / 1e3,
                "expand_roofline_frac": ex_bytes / (hbm_gbs * 1e3) / t_ex,
                "plan_free_expand_us": t_bg,
                "plan_free_form": "no index (one adapter, mask-free)" if single
                                  else "per-token index",
                "torch_mm_us": t_mm, "torch_mm_roofline_frac": mm_bytes / (hbm_gbs * 1e3) / t_mm,
                "pool_sets": n}

    c = li.pages_point()
    r0 = point(c, "SGMV expand m=256 (16x16), r=16, n=2048, 4 adapters sorted, add=0, fp16")
    r0["pages_figures_us"] = {"sgmv_expand": 5.45, "torch_mm": 4.14,
                              "note": "the pages' GPU is not named; context only"}
    res["pages_point"] = r0
    c1 = li.pages_point()
    c1.seg_start = torch.zeros(1, dtype=torch.int32)
    c1.seg_len = torch.full((1,), c1.T, dtype=torch.int32)
    c1.seg_lora = torch.zeros(1, dtype=torch.int32)
    res["single_adapter"] = point(c1, "one adapter, one 256-token segment, r=16, n=2048, "
                                      "add=0, fp16 (the dense special case)")

    shapes = {}
    for name in li.MODEL_SHAPES:
        per_T = {}
        for T in (16, 1024):
            c = li.model_shape(name, T)
            Hm, N, r = c.A.shape[2], c.B[0].shape[1], c.R
            idx = c.token_idx
            act = idx >= 0
            Ta = int(act.sum())
            U = int(torch.unique(idx[act]).numel())
            sh_bytes, ex_bytes = single_slice_work(Ta, T, U, Hm, N, r, add=True)
            A0, B0 = c.A.to(dev), c.B[0].to(dev)
            idx_d = idx.to(dev)

            def mk(i, c=c, A0=A0, B0=B0, idx_d=idx_d, T=T):
                plan = lg.new_plan(T, c.L, dev)
                lg.lora_group_tokens(idx_d, c.L, plan)
                return {"x": c.x.to(dev), "A": A0, "B": B0, "out": c.out.to(dev),
                        "y": torch.zeros(T, r, dtype=torch.float32, device=dev), "plan": plan}

            set_bytes = T * Hm * 2 + T * N * 2 + T * r * 4
            t_sh, n = pool_op_us(mk, lambda a: lg.lora_shrink(a["x"], a["A"], a["y"], a["plan"]),
                                 set_bytes, l2)
            t_ex, _ = pool_op_us(mk, lambda a: lg.lora_expand(a["y"], a["B"], a["out"], a["plan"],
                                                              add_inputs=True), set_bytes, l2)
            per_T[str(T)] = {"H": Hm, "N": N, "shrink_us": t_sh,
                             "shrink_roofline_frac": sh_bytes / (hbm_gbs * 1e3) / t_sh,
                             "expand_us": t_ex,
                             "expand_roofline_frac": ex_bytes / (hbm_gbs * 1e3) / t_ex,
                             "pool_sets": n}
            torch.cuda.synchronize()
        shapes[name] = per_T
    res["model_shapes"] = shapes
    return res


def _device_normal(shape, std, dtype, dev, gen):
    return (torch.randn(shape, generator=gen, device=dev, dtype=torch.float32) * std).to(dtype)


def sweep_work(T: int, Hm: int, N: int, r: int, U: int):
    """Algorithmic bytes of one sweep point (every token active, add_inputs):
    shrink = x + the U used adapters' A rows + y written; expand = y read +
    the used B rows + out read and written."""
    sh_b = T * Hm * 2 + U * r * Hm * 2 + T * r * 4
    ex_b = T * r * 4 + U * N * r * 2 + 2 * T * N * 2
    return sh_b, ex_b


def sweep_rows(lg, dev, hbm_gbs: float, max_sets: int = 256, reps: int = 3):
    """The microbenchmark sweep (vLLM PR #11579's list_bench commands): hidden
    sizes {1024, 2048, 2049, 4096, 8192, 16384} x batch {16 .. 8192} at seq-len
    1 (BGMV, one token per request) and 8 (SGMV, one 8-token segment per
    request), r = 16, 4 adapters drawn uniformly and sorted by id, fp16,
    expand to N = H with add_inputs.  Shrink and expand are timed separately:
    the average launch over a rotating pool of argument sets (>= 4x L2, at
    most `max_sets` sets; `pool_MB` says how much), inputs drawn on the device.
    Seq-len 1 runs the plan-free BGMV operators where they take the shape
    (H % 8 == 0), the grouped ones otherwise; seq-len 8 runs the grouped
    operators on a segment plan built once (outside the timing)."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    gen = torch.Generator(device=dev)
    gen.manual_seed(li.SEED_BASE + 5)
    r, Ls = 16, 4
    rows = []
    for Hm in li.SWEEP_H:
        for batch in li.SWEEP_BATCH:
            for sl in (1, 8):
                T, N = batch * sl, Hm
                ids_req, _ = torch.sort(torch.randint(0, Ls, (batch,), generator=gen, device=dev,
                                                      dtype=torch.int32))
                U = int(torch.unique(ids_req).numel())
                set_bytes = T * Hm * 2 + T * N * 2 + T * r * 4 + 2 * Ls * r * Hm * 2
                nsets = int(min(max_sets, max(1, -(-4 * l2 // set_bytes))))
                sets = [{"x": _device_normal((T, Hm), 1.0, torch.float16, dev, gen),
                         "A": _device_normal((Ls, r, Hm), 0.02, torch.float16, dev, gen),
                         "B": _device_normal((Ls, N, r), 0.02, torch.float16, dev, gen),
                         "out": _device_normal((T, N), 1.0, torch.float16, dev, gen),
                         "y": torch.empty(T, r, device=dev)} for _ in range(nsets)]
                if sl == 1:
                    idx = ids_req.contiguous()
                    path = "bgmv" if Hm % 8 == 0 else "grouped"
                    if path == "grouped":
                        plan = lg.new_plan(T, Ls, dev)
                        lg.lora_group_tokens(idx, Ls, plan)
                else:
                    path = "grouped"
                    plan = lg.new_plan(T, Ls, dev)
                    starts = torch.arange(batch, dtype=torch.int32, device=dev) * sl
                    lens = torch.full((batch,), sl, dtype=torch.int32, device=dev)
                    lg.lora_group_segments(starts, lens, ids_req, T, Ls, plan)
                if path == "bgmv":
                    sh = lambda a: lg.lora_bgmv_shrink(a["x"], a["A"], a["y"], idx)
                    ex = lambda a: lg.lora_bgmv_expand_slice(a["y"], [a["B"]], a["out"], [0], idx,
                                                             y_slice_stride=0, add_inputs=True)
                else:
                    sh = lambda a: lg.lora_shrink(a["x"], a["A"], a["y"], plan)
                    ex = lambda a: lg.lora_expand(a["y"], a["B"], a["out"], plan, add_inputs=True)
                t_sh = _graph_avg_us(sets, sh, reps)
                t_ex = _graph_avg_us(sets, ex, reps)
                sh_b, ex_b = sweep_work(T, Hm, N, r, U)
                rows.append({"H": Hm, "batch": batch, "seq_len": sl, "T": T, "path": path,
                             "shrink_us": round(t_sh, 3),
                             "shrink_frac": round(sh_b / (hbm_gbs * 1e3) / t_sh, 4),
                             "expand_us": round(t_ex, 3),
                             "expand_GBps": round(ex_b / t_ex / 1e3, 1),
                             "expand_frac": round(ex_b / (hbm_gbs * 1e3) / t_ex, 4),
                             "pool_MB": round(nsets * set_bytes / 1e6, 1)})
                del sets
    torch.cuda.synchronize()
    return {"unit": "us per launch; frac = algorithmic bytes / measured HBM bandwidth / time",
            "points": rows}


def _graph_avg_us(sets, launch, reps: int) -> float:
    """Average launch duration: one launch per argument set captured in one
    CUDA graph, replayed `reps` times between two events on its stream."""
    launch(sets[0])
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for a in sets:
            launch(a)
    g.replay()
    # the replays run on torch's current stream, which the events bracket
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(reps):
        g.replay()
    t1.record()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) * 1e3 / (reps * len(sets))


def mixed_rank_rows(lg, dev, hbm_gbs: float, reps: int = 3):
    """The mixed-rank Llama-3-70B-shaped workload: T = 2048, H = 8192, 32
    adapters with ranks from {2, 8, 16, 20, 64, 128} (stored at R = 128), Zipf(1.1)
    adapter per token, 5 % without an adapter, bf16, expand to N in {8192,
    28672}, BGMV (token order) and SGMV (tokens sorted into segments).  The
    rank-aware call (the ranks table: rows / columns past a rank never read)
    is timed against padding every adapter to rank 128 (no ranks table, the
    padding zero-filled), the workaround Punica issue #17 describes.  Each
    figure: average launch over a rotating pool >= 4x L2; tensors on the
    device."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    gen = torch.Generator(device=dev)
    gen.manual_seed(li.SEED_BASE + 4)
    T, Hm, L = 2048, 8192, 32
    res = {}
    for sgmv in (False, True):
        ranks, mp = li.mixed_rank_map(T=T, L=L, sgmv=sgmv)
        R = int(ranks.max())
        plan = lg.new_plan(T, L, dev)
        if sgmv:
            ss, sl_, so = (t.to(dev) for t in mp)
            lg.lora_group_segments(ss, sl_, so, T, L, plan)
            lora_of = torch.repeat_interleave(so.cpu(), sl_.cpu())
        else:
            lg.lora_group_tokens(mp.to(dev), L, plan)
            lora_of = mp
        act = lora_of >= 0
        Ta = int(act.sum())
        used = torch.unique(lora_of[act]).long()
        r_used = int(ranks[used].sum())
        r_tok = int(ranks[lora_of[act].long()].sum())
        ranks_d = ranks.to(dev)
        keep = (torch.arange(R)[None, :] < ranks[:, None]).to(dev)  # [L, R]
        for N in (8192, 28672):
            set_bytes = T * Hm * 2 + L * R * Hm * 2 + L * N * R * 2 + T * N * 2 + T * R * 4
            nsets = int(max(1, -(-4 * l2 // set_bytes)))
            sets = []
            for _ in range(nsets):
                A = _device_normal((L, R, Hm), 0.02, torch.bfloat16, dev, gen) * keep[:, :, None]
                B = _device_normal((L, N, R), 0.02, torch.bfloat16, dev, gen) * keep[:, None, :]
                sets.append({"x": _device_normal((T, Hm), 1.0, torch.bfloat16, dev, gen),
                             "A": A.contiguous(), "B": B.contiguous(),
                             "out": _device_normal((T, N), 1.0, torch.bfloat16, dev, gen),
                             "y": torch.zeros(T, R, device=dev)})
            row = {"N": N, "pool_sets": nsets}
            for tag, rk in (("rank_aware", ranks_d), ("padded_to_128", None)):
                t_sh = _graph_avg_us(sets, lambda a: lg.lora_shrink(a["x"], a["A"], a["y"], plan,
                                                                     ranks=rk), reps)
                t_ex = _graph_avg_us(sets, lambda a: lg.lora_expand(a["y"], a["B"], a["out"], plan,
                                                                     ranks=rk, add_inputs=True),
                                     reps)
                ru, rt = (r_used, r_tok) if rk is not None else (len(used) * R, Ta * R)
                sh_b = Ta * Hm * 2 + ru * Hm * 2 + T * R * 4
                ex_b = rt * 4 + ru * N * 2 + 2 * Ta * N * 2
                row[tag] = {"shrink_us": round(t_sh, 2),
                            "shrink_frac": round(sh_b / (hbm_gbs * 1e3) / t_sh, 4),
                            "expand_us": round(t_ex, 2),
                            "expand_frac": round(ex_b / (hbm_gbs * 1e3) / t_ex, 4),
                            "bytes": {"shrink": sh_b, "expand": ex_b}}
            row["speedup_rank_aware"] = round(
                (row["padded_to_128"]["shrink_us"] + row["padded_to_128"]["expand_us"]) /
                (row["rank_aware"]["shrink_us"] + row["rank_aware"]["expand_us"]), 3)
            res[f"{'sgmv' if sgmv else 'bgmv'}_N{N}"] = row
            del sets
    torch.cuda.synchronize()
    res["ranks"] = ranks.tolist()
    return res


def algorithmic_fused(idx: torch.Tensor):
    """Fused shrink + expand_slice: x, live A rows, y written once, live B
    rows, out read and written (y is not re-read from HBM)."""
    sb, sf, eb, ef = algorithmic(idx)
    Ta = int((idx >= 0).sum())
    return sb + eb - Ta * len(SLICES) * R * 4, sf + ef


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=5)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- our arm

def make_pool(dev, rank: int, l2_bytes: int, only_T=None):
    """Rotating argument pool: sets of (inputs, adapters, outputs) for every
    batch size, enough sets that the pool is >= 4x L2, so each step reads
    data no earlier step left in L2."""
    import lora_gemv_gb300 as lg
    per_set = 0
    for T in li.DECODE_T:
        per_set += T * (H * E + NTOT * E + len(SLICES) * R * 4 + 4) + L * (len(SLICES) * R * H
                                                                            + NTOT * R) * E
    nsets = max(2, -(-4 * l2_bytes // per_set)) if only_T is None else 1
    pool = []
    for s in range(nsets):
        batches = []
        for T in (li.DECODE_T if only_T is None else (only_T,)):
            c = li.decode_qkv(T, seed=li.SEED_BASE + 2 + 1000 * rank + 17 * s + T)
            batches.append({
                "T": T, "case": c,
                "x": c.x.to(dev), "A": c.A.to(dev), "B": [b.to(dev) for b in c.B],
                "out": c.out.to(dev), "idx": c.token_idx.to(dev),
                "y": torch.empty(T, len(SLICES) * R, dtype=torch.float32, device=dev),
                "plan": lg.new_plan(T, L, dev),
            })
        pool.append(batches)
    return pool, nsets * per_set



# DRAM bytes (read + write) of one launch of each kernel for the T=1024 batch,
# from an ncu capture of `bench.py --profile --T 1024` (summaries under
# profiles/); None until a capture of the current kernel exists.
NCU_TRAFFIC = {
    "shrink": {"bytes": 9177856, "source": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum: "
               "9.178 MB read + 0 written (y stays in L2), T=1024 launch of the current "
               "tcgen05 variant without TMA staging"},
}


# The decode step's path: "grouped" = BGMV grouping into a plan, then the
# chained grouped operators (the faster of the two on the decode step);
# "bgmv" = the plan-free operators (no grouping; the stacked q/k/v shrink and
# the three-slice expand chained in one call), timed beside it.
STEP_PATH = "grouped"
# "hybrid": the plan-free operators for batches of at most HYBRID_MAX_T tokens
# (where they match the grouped path and save the grouping launch), the
# grouped ones above
HYBRID_MAX_T = 256
LAUNCHES_PER_BATCH = {"bgmv": 2, "grouped": 3}


def step_launches(path: str) -> int:
    """Kernel launches of one decode step (all five batches) on `path`."""
    if path == "hybrid":
        return sum(2 if T <= HYBRID_MAX_T else 3 for T in li.DECODE_T)
    return LAUNCHES_PER_BATCH[path] * len(li.DECODE_T)


def run_step(lg, batches, path: str = STEP_PATH):
    """One decode step over `batches` (q/k/v shrink and expand_slice per batch)."""
    for b in batches:
        if path == "bgmv" or (path == "hybrid" and b["T"] <= HYBRID_MAX_T):
            lg.lora_bgmv_shrink_expand_slice(b["x"], b["A"], b["y"], b["B"], b["out"],
                                             b["case"].slice_offsets, b["idx"], add_inputs=True)
        else:
            lg.lora_group_tokens(b["idx"], L, b["plan"])
            lg.lora_shrink_expand_slice(b["x"], b["A"], b["y"], b["B"], b["out"], b["plan"],
                                        b["case"].slice_offsets, add_inputs=True)


def e2e_run(lg, dev, steps: int, warmup: int, path: str = "bgmv"):
    """Through the public API with host buffers.  Every step uploads the five
    batches' inputs (x, token indices, base output) from pinned host memory,
    runs the path and downloads the updated outputs.  The inputs are packed
    in one pinned buffer and one device buffer laid out [all x | all
    indices | all out], so a step is one host-to-device copy, the path's
    calls on views of that buffer, and one device-to-host copy of the out
    region.  Two such buffers alternate: the upload of step k+1 (copy stream)
    overlaps the compute of step k, and the download of step k (a second
    copy stream) overlaps both.  Returns tokens/s from CUDA events around the
    timed steps, the bytes each way per step, wall-clock tokens/s and the
    host link's copy bandwidth measured alone (same buffers)."""
    align = 256
    cases = [li.decode_qkv(T, seed=li.SEED_BASE + 2 + 5 * T) for T in li.DECODE_T]
    offs, pos = [], 0

    def take(nbytes):
        nonlocal pos
        o = pos
        pos = (pos + nbytes + align - 1) // align * align
        return o

    x_off = [take(c.x.numel() * 2) for c in cases]
    i_off = [take(c.token_idx.numel() * 4) for c in cases]
    out_begin = pos
    o_off = [take(c.out.numel() * 2) for c in cases]
    total, out_bytes = pos, pos - out_begin
    slots = []
    for _ in range(2):
        hin = torch.empty(total, dtype=torch.uint8).pin_memory()
        for c, xo, io, oo in zip(cases, x_off, i_off, o_off):
            hin[xo:xo + c.x.numel() * 2].copy_(c.x.reshape(-1).view(torch.uint8))
            hin[io:io + c.token_idx.numel() * 4].copy_(c.token_idx.view(torch.uint8))
            hin[oo:oo + c.out.numel() * 2].copy_(c.out.reshape(-1).view(torch.uint8))
        dbuf = torch.empty(total, dtype=torch.uint8, device=dev)
        batches = []
        for c, xo, io, oo in zip(cases, x_off, i_off, o_off):
            T = c.T
            batches.append({
                "T": T, "case": c,
                "x": dbuf[xo:xo + T * H * 2].view(torch.bfloat16).view(T, H),
                "idx": dbuf[io:io + T * 4].view(torch.int32),
                "out": dbuf[oo:oo + T * NTOT * 2].view(torch.bfloat16).view(T, NTOT),
                "y": torch.empty(T, len(SLICES) * R, dtype=torch.float32, device=dev),
                "plan": lg.new_plan(T, L, dev)})
        slots.append({"hin": hin, "hout": torch.empty(out_bytes, dtype=torch.uint8).pin_memory(),
                      "dbuf": dbuf, "batches": batches,
                      "up": torch.cuda.Event(), "done": torch.cuda.Event(),
                      "down": torch.cuda.Event()})
    weights = [{"A": c.A.to(dev), "B": [b.to(dev) for b in c.B]} for c in cases]
    for sl in slots:
        for b, w in zip(sl["batches"], weights):
            b.update(w)
    comp = torch.cuda.current_stream(dev)
    up_s, down_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    for sl in slots:
        sl["down"].record(down_s)

    def step(k):
        sl = slots[k % 2]
        up_s.wait_event(sl["down"])       # the slot's previous outputs are downloaded
        with torch.cuda.stream(up_s):
            sl["dbuf"].copy_(sl["hin"], non_blocking=True)
        sl["up"].record(up_s)
        comp.wait_event(sl["up"])
        run_step(lg, sl["batches"], path=path)
        sl["done"].record(comp)
        down_s.wait_event(sl["done"])
        with torch.cuda.stream(down_s):
            sl["hout"].copy_(sl["dbuf"][out_begin:], non_blocking=True)
        sl["down"].record(down_s)

    for k in range(warmup):
        step(k)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    t0.record(up_s)
    for k in range(steps):
        step(warmup + k)
    t1.record(down_s)
    torch.cuda.synchronize()
    wall = time.perf_counter() - w0
    ms = t0.elapsed_time(t1)
    tokens = steps * sum(li.DECODE_T)
    # the host link alone: the same upload and download, back to back
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(up_s):
        c0.record(up_s)
        for k in range(20):
            slots[k % 2]["dbuf"].copy_(slots[k % 2]["hin"], non_blocking=True)
        c1.record(up_s)
    torch.cuda.synchronize()
    h2d_gbs = 20 * total / (c0.elapsed_time(c1) / 1e3) / 1e9
    with torch.cuda.stream(down_s):
        c0.record(down_s)
        for k in range(20):
            slots[k % 2]["hout"].copy_(slots[k % 2]["dbuf"][out_begin:], non_blocking=True)
        c1.record(down_s)
    torch.cuda.synchronize()
    d2h_gbs = 20 * out_bytes / (c0.elapsed_time(c1) / 1e3) / 1e9
    return tokens / (ms / 1e3), total, out_bytes, tokens / wall, h2d_gbs, d2h_gbs


def cpu_baseline(target_s: float = 10.0):
    """The oracle, as it stands, on the same decode batches on the host cores:
    with every core (OpenMP over tokens; the reported figure) and on one
    thread (beside it), each for about target_s / 2 seconds of whole steps."""
    import oracle
    prepared = []
    for T in li.DECODE_T:
        c = li.decode_qkv(T)
        prepared.append((T, c.token_idx.numpy(), c.x.double().numpy(), c.A.double().numpy(),
                         [b.double().numpy() for b in c.B], c.out.double().numpy(),
                         c.slice_offsets))

    def run(seconds):
        tokens, reps = 0, 0
        t0 = time.perf_counter()
        while True:
            for T, idx, x, A, Bs, out, offs in prepared:
                lo, _ = oracle.map_tokens(idx, L)
                y = oracle.shrink(x, A, lo, num_slices=len(SLICES))
                oracle.expand_slice(y, Bs, offs, lo, out, y_stride=R, add=True)
                tokens += T
            reps += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                return tokens, reps, el

    cores = oracle.num_threads()
    tokens, reps, el = run(target_s / 2)
    oracle.set_threads(1)
    t1, r1, e1 = run(target_s / 2)
    oracle.set_threads(cores)
    return {"value": tokens / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "one_thread": {"value": t1 / e1, "unit": "tokens/s", "cores": 1,
                           "sample": f"{r1} full steps, {e1:.1f} s"},
            "sample": f"{reps} full steps ({tokens} tokens of the same five decode batches), "
                      f"fp64 C loops, OpenMP over tokens, {el:.1f} s"}


def capture_steps(lg, pool, concurrent: bool, path: str = STEP_PATH):
    """One CUDA graph per pool set holding a whole step (launch overhead off
    the timed path, as the pages time their kernels).  With `concurrent` the
    step's independent decode batches are parallel branches of the graph
    (fork/join on side streams), so the latency-bound small batches overlap
    the large ones; otherwise they run one after another.  The graphs hold no
    event nodes: on this GPU an event-record node costs several microseconds,
    far more than the decode kernels themselves."""
    graphs = []
    stream = torch.cuda.Stream()
    side = [torch.cuda.Stream() for _ in li.DECODE_T]
    for batches in pool:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            if concurrent:
                fork = torch.cuda.Event()
                fork.record(stream)
                joins = []
                for b, st in zip(batches, side):
                    st.wait_event(fork)
                    with torch.cuda.stream(st):
                        run_step(lg, [b], path=path)
                    ev = torch.cuda.Event()
                    ev.record(st)
                    joins.append(ev)
                for ev in joins:
                    stream.wait_event(ev)
            else:
                run_step(lg, batches, path=path)
        graphs.append(g)
    torch.cuda.synchronize()
    return graphs


def time_graphs(graphs, W: int, K: int):
    for w in range(W):
        graphs[w % len(graphs)].replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    for k in range(K):
        graphs[(W + k) % len(graphs)].replay()
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def op_only_ms(pool, launch, reps: int = 20, max_T: Optional[int] = None):
    """Average duration of one operator per batch size: a graph of one launch
    per pool set (each on a different set, so inputs come from HBM), replayed
    `reps` times between two events on the launching stream.  Batch sizes
    above `max_T` get None."""
    res = []
    stream = torch.cuda.Stream()
    for i in range(len(li.DECODE_T)):
        if max_T is not None and li.DECODE_T[i] > max_T:
            res.append(None)
            continue
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for batches in pool:
                launch(batches[i])
        g.replay()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(reps):
            g.replay()
        t1.record()
        torch.cuda.synchronize()
        res.append(t0.elapsed_time(t1) / (reps * len(pool)))
    return res


def expand_only_ms(lg, pool, reps: int = 20):
    """Average duration of expand_slice per batch size: a graph of one launch
    per pool set (each on a different set, so inputs come from HBM), replayed
    `reps` times between two events on the launching stream."""
    res = []
    stream = torch.cuda.Stream()
    for i in range(len(li.DECODE_T)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for batches in pool:
                b = batches[i]
                lg.lora_expand_slice(b["y"], b["B"], b["out"], b["plan"],
                                     b["case"].slice_offsets, y_slice_stride=R, add_inputs=True)
        g.replay()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(reps):
            g.replay()
        t1.record()
        torch.cuda.synchronize()
        res.append(t0.elapsed_time(t1) / (reps * len(pool)))
    return res


def main_ours(args):
    import torch.distributed as dist
    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import lora_gemv_gb300 as lg
    lg.load()
    props = torch.cuda.get_device_properties(dev)
    pool, pool_bytes = make_pool(dev, rank, props.L2_cache_size)
    nsets = len(pool)
    K, W = args.steps, args.warmup

    others = [p for p in ("grouped", "bgmv", "hybrid") if p != STEP_PATH]
    for w in range(max(W, 1)):  # eager warm-up also configures the kernels before capture
        run_step(lg, pool[w % nsets])
        for p_ in others:
            run_step(lg, pool[w % nsets], path=p_)
    torch.cuda.synchronize()
    graphs = capture_steps(lg, pool, concurrent=True)
    seq_graphs = capture_steps(lg, pool, concurrent=False)
    other_graphs = {p_: capture_steps(lg, pool, concurrent=True, path=p_) for p_ in others}
    for w in range(W):
        graphs[w % nsets].replay()
    torch.cuda.synchronize()

    nb = len(li.DECODE_T)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    cvd = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    clocks = ClockSampler(int(cvd.split(",")[local]) if cvd and all(
        c.strip().isdigit() for c in cvd.split(",")) else local)
    clocks.start()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    start.record()
    for k in range(K):
        graphs[(W + k) % nsets].replay()
    end.record()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()

    ms = start.elapsed_time(end)
    seq_ms = time_graphs(seq_graphs, W, K)      # the same steps with the batches in sequence
    # the same steps through the other paths
    other_ms = {p_: time_graphs(g_, W, K) for p_, g_ in other_graphs.items()}

    # per batch size: the chained pair and its kernels alone, on both paths
    offs = pool[0][0]["case"].slice_offsets
    times = {
        "grouped": {
            "pair": op_only_ms(pool, lambda b: lg.lora_shrink_expand_slice(
                b["x"], b["A"], b["y"], b["B"], b["out"], b["plan"], offs, add_inputs=True)),
            "shrink": op_only_ms(pool, lambda b: lg.lora_shrink(b["x"], b["A"], b["y"], b["plan"],
                                                                num_slices=len(SLICES))),
            "expand_slice": expand_only_ms(lg, pool),
            "grouping": op_only_ms(pool, lambda b: lg.lora_group_tokens(b["idx"], L, b["plan"])),
        },
        "bgmv": {
            "pair": op_only_ms(pool, lambda b: lg.lora_bgmv_shrink_expand_slice(
                b["x"], b["A"], b["y"], b["B"], b["out"], offs, b["idx"], add_inputs=True)),
            "shrink": op_only_ms(pool, lambda b: lg.lora_bgmv_shrink(
                b["x"], b["A"], b["y"], b["idx"], num_slices=len(SLICES))),
            "expand_slice": op_only_ms(pool, lambda b: lg.lora_bgmv_expand_slice(
                b["y"], b["B"], b["out"], offs, b["idx"], y_slice_stride=R, add_inputs=True)),
        },
    }
    # the same decode pair as one cooperative launch (batches of at most 256 tokens)
    fused_ms = op_only_ms(pool, lambda b: lg.lora_bgmv_fused_shrink_expand_slice(
        b["x"], b["A"], b["y"], b["B"], b["out"], offs, b["idx"], add_inputs=True),
        max_T=lg.FUSED_MAX_TOKENS)
    ex_src = (f"CUDA events around graphs of back-to-back launches, one per pool set "
              f"({nsets} sets, inputs from HBM), per batch size")
    tokens_rank = K * sum(li.DECODE_T)
    ms, _, value = aggregate(ms, tokens_rank, ws, dev)

    per_T = {}
    pair_bytes = 0
    for i, T in enumerate(li.DECODE_T):
        idx = pool[0][i]["case"].token_idx
        sb, sf, eb, ef = algorithmic(idx)
        fb, ff = algorithmic_fused(idx)
        pair_bytes += fb
        row = {"shrink_bytes": sb, "expand_bytes": eb, "pair_bytes": fb}
        for path, tk in times.items():
            row[path] = {f"{k}_us": v[i] * 1e3 for k, v in tk.items()}
            row[path]["shrink_GBps"] = sb / (tk["shrink"][i] / 1e3) / 1e9
            row[path]["expand_GBps"] = eb / (tk["expand_slice"][i] / 1e3) / 1e9
        if fused_ms[i] is not None:
            row["fused_one_launch"] = {"pair_us": fused_ms[i] * 1e3,
                                       "pair_GBps": fb / (fused_ms[i] / 1e3) / 1e9}
        per_T[str(T)] = row
    hbm, tf, src = peaks()
    # dominant kernel: the largest summed per-step time among the operators of
    # the path that runs the largest batch; its roofline is taken on its launch
    # for the largest batch (algorithmic bytes of that launch / its measured
    # duration), with the all-batch figure beside it
    big_path = "grouped" if STEP_PATH in ("grouped", "hybrid") else "bgmv"
    tk = times[big_path]
    byte_key = {"shrink": "shrink_bytes", "expand_slice": "expand_bytes"}
    dom = max(byte_key, key=lambda k: sum(tk[k]))
    dom_ms, dom_key = tk[dom], byte_key[dom]
    Tmax = str(li.DECODE_T[-1])
    achieved = per_T[Tmax][dom_key] / (dom_ms[-1] / 1e3) / 1e9
    all_achieved = sum(v[dom_key] for v in per_T.values()) / (sum(dom_ms) / 1e3) / 1e9
    step_s = ms / 1e3 / K
    path_frac = (pair_bytes / (hbm * 1e9)) / step_s
    dom_name = dom if big_path == "grouped" else f"bgmv_{dom}"
    traffic = NCU_TRAFFIC.get(dom_name)
    kernels = [k for k in tk if k != "pair"]

    e2e_v, h2d, d2h, e2e_wall, h2d_gbs, d2h_gbs = e2e_run(lg, dev, max(10, min(K, 300)), 3)

    res = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K,
        "warmup": W, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, shapes of the workload)",
        "config": {"workload": WORKLOAD, "tokens_per_step_per_gpu": sum(li.DECODE_T),
                   "parallelism": f"replicas x{ws} (independent batches, no collective)",
                   "l2": f"rotating argument pool of {nsets} sets ({pool_bytes / 1e6:.0f} MB "
                         f">= 4x L2 {props.L2_cache_size / 1e6:.0f} MB): inputs larger than L2",
                   "launch": "each step replayed from a CUDA graph (one per pool set); the "
                             "five independent batches are concurrent branches of the graph",
                   "path": STEP_PATH},
        "sequential_batches": {"value": tokens_rank * ws / (seq_ms / 1e3), "unit": "tokens/s",
                               "ms_per_step": seq_ms / K},
        "other_paths": {p_: {"value": tokens_rank * ws / (m_ / 1e3), "unit": "tokens/s",
                             "ms_per_step": m_ / K} for p_, m_ in other_ms.items()},
        "paths": {"grouped": "lora_group_tokens + the chained grouped operators, 3 launches "
                             "per batch",
                  "bgmv": "the chained plan-free operators, 2 launches per batch",
                  "hybrid": f"bgmv for T <= {HYBRID_MAX_T}, grouped above"},
        "roofline": {"kernel": dom_name, "launch": f"T={Tmax} batch", "bound": "hbm",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "peak_source": f"{src} hbm_gbs",
                     "traffic": traffic["bytes"] if traffic else None,
                     "traffic_source": traffic["source"] if traffic else None,
                     "all_batches_achieved": all_achieved, "timing": ex_src},
        "step_time_share": {k: sum(tk[k]) / sum(sum(tk[q]) for q in kernels) for k in kernels},
        "path_roofline_frac": path_frac,
        # per batch: (grouping,) shrink and expand_slice
        "gpu_launches": K * step_launches(STEP_PATH),
        "e2e": {"value": e2e_v, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "wall_tokens_per_s": e2e_wall,
                "host_link_GBps": {"h2d": h2d_gbs, "d2h": d2h_gbs},
                "how": "public Python API per call (no graph); each step one packed upload "
                       "from pinned memory and one download of the outputs, double-buffered "
                       "on copy streams"},
        "clocks": clk,
        "per_T": per_T,
        "prefill_sgmv": prefill_sgmv(lg, dev, hbm, tf),
        "next_rows": next_rows(lg, dev, hbm),
        "wall_s_timed": wall,
    }
    if not args.quick:
        res["mixed_rank"] = mixed_rank_rows(lg, dev, hbm)
        res["sweep"] = sweep_rows(lg, dev, hbm)
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    prepared = []
    for T in li.DECODE_T:
        c = li.decode_qkv(T)
        prepared.append((T, c.token_idx.numpy(), c.x.double().numpy(), c.A.double().numpy(),
                         [b.double().numpy() for b in c.B], c.out.double().numpy(),
                         c.slice_offsets))
    # Bounded sample per step: a slice of each batch's tokens, sized so the
    # whole run stays within about two minutes.
    budget = float(args.ref_budget_s)
    t0 = time.perf_counter()
    _ref_step(oracle, prepared, None)
    full = time.perf_counter() - t0
    frac = min(1.0, budget / max(1e-6, full * (args.steps + args.warmup)))
    rows = {T: max(1, int(round(T * frac))) for T in li.DECODE_T}
    for _ in range(args.warmup):
        _ref_step(oracle, prepared, rows)
    t0 = time.perf_counter()
    tokens = 0
    for _ in range(args.steps):
        tokens += _ref_step(oracle, prepared, rows)
    el = time.perf_counter() - t0
    v = tokens / el
    res = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": ws,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded, shapes of the workload)",
           "config": {"workload": WORKLOAD, "tokens_per_step_sampled": sum(rows.values())},
           "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": oracle.num_threads(),
                            "kind": "oracle",
                            "sample": f"first {rows} tokens of each decode batch per step"},
           "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def _ref_step(oracle, prepared, rows):
    n = 0
    for T, idx, x, A, Bs, out, offs in prepared:
        k = T if rows is None else rows[T]
        lo, _ = oracle.map_tokens(idx[:k], L)
        y = oracle.shrink(x[:k], A, lo, num_slices=len(SLICES))
        oracle.expand_slice(y, Bs, offs, lo, out[:k], y_stride=R, add=True)
        n += k
    return n


def main_profile(args):
    """A few eager launches of the path (--path) on one decode batch, for
    profilers (e.g. ncu -k regex:expand -s 2 -c 1 python bench.py --profile --T 1024),
    or with --prefill-r R on the prefill gate/up workload at rank R (grouping,
    shrink, expand_slice per repetition)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import lora_gemv_gb300 as lg
    lg.load()
    if args.prefill_r:
        r = args.prefill_r
        c = li.prefill_gateup(r=r)
        x, A = c.x.to(dev), c.A.to(dev)
        Bs = [b.to(dev) for b in c.B]
        out = c.out.to(dev)
        y = torch.empty(c.T, c.num_slices * r, dtype=torch.float32, device=dev)
        plan = lg.new_plan(c.T, c.L, dev)
        ss, sl, slo = c.seg_start.to(dev), c.seg_len.to(dev), c.seg_lora.to(dev)
        for _ in range(args.profile_reps):
            lg.lora_group_segments(ss, sl, slo, c.T, c.L, plan)
            lg.lora_shrink(x, A, y, plan, num_slices=c.num_slices)
            lg.lora_expand_slice(y, Bs, out, plan, c.slice_offsets, y_slice_stride=r,
                                 add_inputs=True)
        torch.cuda.synchronize()
        print(json.dumps({"profile": True, "workload": "prefill_gateup", "r": r, "T": c.T,
                          "reps": args.profile_reps}))
        return
    if args.sweep_point:
        # one point of the hidden-size x batch sweep: grouping, shrink, expand
        Hs, bs, sls = (int(v) for v in args.sweep_point.split(","))
        c = li.sweep(Hs, bs, sls)
        x, A, B, out = c.x.to(dev), c.A.to(dev), c.B[0].to(dev), c.out.to(dev)
        y = torch.empty(c.T, c.R, dtype=torch.float32, device=dev)
        plan = lg.new_plan(c.T, c.L, dev)
        for _ in range(args.profile_reps):
            if sls == 1:
                lg.lora_group_tokens(c.token_idx.to(dev), c.L, plan)
            else:
                lg.lora_group_segments(c.seg_start.to(dev), c.seg_len.to(dev), c.seg_lora.to(dev),
                                       c.T, c.L, plan)
            lg.lora_shrink(x, A, y, plan)
            lg.lora_expand(y, B, out, plan, add_inputs=True)
        torch.cuda.synchronize()
        print(json.dumps({"profile": True, "workload": "sweep", "H": Hs, "batch": bs,
                          "seq_len": sls, "T": c.T, "reps": args.profile_reps}))
        return
    if args.path == "single":
        # one adapter, no token index (the mask-free dense expand), at T rows
        g = torch.Generator().manual_seed(li.SEED_BASE + 77)
        y = torch.randn(args.T, 16, generator=g).to(dev)
        B = (torch.randn(1, 2048, 16, generator=g) * 0.02).half().to(dev)
        out = torch.empty(args.T, 2048, dtype=torch.float16, device=dev)
        for _ in range(args.profile_reps):
            lg.lora_bgmv_expand_slice(y, [B], out, [0], None, y_slice_stride=0, add_inputs=False)
        torch.cuda.synchronize()
        print(json.dumps({"profile": True, "path": "single", "T": args.T, "N": 2048, "r": 16,
                          "reps": args.profile_reps}))
        return
    pool, _ = make_pool(dev, 0, 0, only_T=args.T)
    offs = pool[0][0]["case"].slice_offsets
    for _ in range(args.profile_reps):
        for batches in pool:
            if args.path == "fused":
                for b in batches:
                    lg.lora_bgmv_fused_shrink_expand_slice(b["x"], b["A"], b["y"], b["B"], b["out"],
                                                           offs, b["idx"], add_inputs=True)
            else:
                run_step(lg, batches, path=args.path)
    torch.cuda.synchronize()
    print(json.dumps({"profile": True, "path": args.path, "T": args.T,
                      "reps": args.profile_reps}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true",
                    help="skip the mixed-rank and sweep sections")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-budget-s", type=float, default=90.0)
    ap.add_argument("--profile", action="store_true",
                    help="run a few eager steps of one decode batch (for ncu), no timing")
    ap.add_argument("--T", type=int, default=1024, help="batch size for --profile")
    ap.add_argument("--profile-reps", type=int, default=3)
    ap.add_argument("--path", choices=["grouped", "bgmv", "fused", "single"], default=STEP_PATH,
                    help="with --profile: the decode pair's path (single: the one-adapter "
                         "expand at T x 2048, r = 16)")
    ap.add_argument("--sweep-point", default="",
                    help="with --profile: one sweep point 'H,batch,seq_len' (grouped path)")
    ap.add_argument("--prefill-r", type=int, default=0,
                    help="with --profile: the prefill gate/up workload at this rank instead")
    args = ap.parse_args()
    if args.profile:
        return main_profile(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        main_reference(args)
    else:
        main_ours(args)


if __name__ == "__main__":
    main()
