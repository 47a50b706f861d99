"""Seeded synthetic inputs for the multi-LoRA shrink / expand workloads.

This module only draws random numbers and lays them out; it holds none of
the method's arithmetic.  Both the CUDA path (tests, bench) and the CPU
oracle read the tensors it returns, so they see identical inputs.

All tensors are created on the CPU with a ``torch.Generator`` seeded per
workload, then cast to the workload dtype.  Shapes follow the workloads the
vLLM LoRA microbenchmark PR (#11579) sweeps and the Llama-3 layer shapes its
``model_bench`` mode names:

* ``bgmv_small``     T=16, H=N=1024, r=16, L=4, fp16, idx uniform in {-1..3}
* ``decode_qkv``     Llama-3-8B q/k/v: H=4096, slices 4096/1024/1024, r=16,
                     L=4, bf16, 10 % of tokens idx=-1, the rest uniform
* ``prefill_gateup`` 8 segments, lengths log-uniform in [8, 2048], adapters
                     [0,0,0,1,2,2,3,3] (the "AAABCC" sharing of Punica
                     issue #17), H=4096, gate/up slices of 14336, fp16
* ``mixed_rank_70b`` Llama-3-70B-shaped: H=8192, N in {8192, 28672}, 32
                     adapters with ranks from {2,8,16,20,64,128}, T=2048,
                     Zipf(1.1) adapter popularity, 5 % idx=-1, bf16
* ``sweep``          H in {1024,2048,2049,4096,8192,16384}, batch in
                     {16..8192}, seq-len 1 (BGMV, sorted ids) or 8 (SGMV,
                     one 8-token segment per request, sorted), r=16, L=4, fp16
* ``pages_point``    the single kernel timing the microbenchmark PR prints:
                     SGMV expand, m = 256 tokens (16 requests x 16 tokens),
                     r = 16, n = 2048, 4 adapters, requests sorted by adapter
                     id, add_inputs=False, fp16
* ``model_shape``    Llama-3 projections besides q/k/v and gate/up (o_proj and
                     down_proj, H and N as the layer's input and output
                     widths), decode batches as ``decode_qkv``, one slice

Weights are N(0, 0.02^2) (std 0.02), activations and the base output N(0, 1).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

WEIGHT_STD = 0.02
SEED_BASE = 1000

DECODE_T = (16, 128, 256, 512, 1024)
QKV_SLICES = (4096, 1024, 1024)
GATEUP_N = 14336
SWEEP_H = (1024, 2048, 2049, 4096, 8192, 16384)
SWEEP_BATCH = (16, 128, 256, 512, 1024, 2048, 8192)
MIXED_RANKS = (2, 8, 16, 20, 64, 128)
# (H, N) of the Llama-3 o_proj / down_proj layers (input width, output width)
MODEL_SHAPES = {
    "llama3_8b_o_proj": (4096, 4096),
    "llama3_8b_down_proj": (14336, 4096),
    "llama3_70b_o_proj": (8192, 8192),
    "llama3_70b_down_proj": (28672, 8192),
}


@dataclass
class Case:
    """One shrink + expand(_slice) problem, all tensors on the CPU."""
    name: str
    dtype: torch.dtype
    x: torch.Tensor                  # [T, H]
    A: torch.Tensor                  # [L, S*R, H]  (S stacked slices of R rows)
    B: List[torch.Tensor]            # per slice [L, N_s, R]
    out: torch.Tensor                # [T, N_total] base output (add_inputs=True)
    slice_offsets: List[int]
    R: int                           # rows per slice (= max rank)
    num_slices: int
    L: int
    token_idx: Optional[torch.Tensor] = None    # [T] int32 (BGMV)
    seg_start: Optional[torch.Tensor] = None    # [S] int32 (SGMV)
    seg_len: Optional[torch.Tensor] = None
    seg_lora: Optional[torch.Tensor] = None
    ranks: Optional[torch.Tensor] = None        # [L] int32 or None (all R)
    scale: float = 1.0
    shrink_scale: float = 1.0
    add: bool = True
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return self.x.shape[0]

    @property
    def H(self) -> int:
        return self.x.shape[1]

    @property
    def N_total(self) -> int:
        return self.out.shape[1]

    def lora_of_token(self) -> torch.Tensor:
        """Per-token adapter id as drawn (-1 = none); host-side convenience."""
        if self.token_idx is not None:
            return self.token_idx.clone()
        t = torch.full((self.T,), -1, dtype=torch.int32)
        for s, n, l in zip(self.seg_start.tolist(), self.seg_len.tolist(),
                           self.seg_lora.tolist()):
            t[s:s + n] = l
        return t


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _normal(g, shape, std, dtype):
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(dtype)


def _exact_inactive(g, T: int, frac: float) -> torch.Tensor:
    """Boolean mask with exactly round(frac*T) True entries at seeded positions."""
    k = int(round(frac * T))
    mask = torch.zeros(T, dtype=torch.bool)
    if k:
        mask[torch.randperm(T, generator=g)[:k]] = True
    return mask


def _segments_from_sorted(ids: torch.Tensor):
    """Run-length segments of a per-token id vector (ids already in order)."""
    starts, lens, loras = [], [], []
    T = ids.numel()
    t = 0
    vals = ids.tolist()
    while t < T:
        u = t
        while u < T and vals[u] == vals[t]:
            u += 1
        starts.append(t)
        lens.append(u - t)
        loras.append(vals[t])
        t = u
    i32 = torch.int32
    return torch.tensor(starts, dtype=i32), torch.tensor(lens, dtype=i32), torch.tensor(loras, dtype=i32)


def bgmv_small(seed: int = SEED_BASE + 1, T: int = 16, H: int = 1024, N: int = 1024,
               r: int = 16, L: int = 4, dtype=torch.float16) -> Case:
    g = _gen(seed)
    x = _normal(g, (T, H), 1.0, dtype)
    A = _normal(g, (L, r, H), WEIGHT_STD, dtype)
    B = _normal(g, (L, N, r), WEIGHT_STD, dtype)
    idx = torch.randint(-1, L, (T,), generator=g, dtype=torch.int32)
    out = _normal(g, (T, N), 1.0, dtype)
    return Case("bgmv_small", dtype, x, A, [B], out, [0], r, 1, L, token_idx=idx,
                scale=0.5, add=True)


def decode_qkv(T: int, seed: Optional[int] = None, H: int = 4096, r: int = 16, L: int = 4,
               slices=QKV_SLICES, dtype=torch.bfloat16, inactive: float = 0.10) -> Case:
    g = _gen(SEED_BASE + 2 if seed is None else seed)
    S = len(slices)
    x = _normal(g, (T, H), 1.0, dtype)
    A = _normal(g, (L, S * r, H), WEIGHT_STD, dtype)
    B = [_normal(g, (L, n, r), WEIGHT_STD, dtype) for n in slices]
    idx = torch.randint(0, L, (T,), generator=g, dtype=torch.int32)
    idx[_exact_inactive(g, T, inactive)] = -1
    out = _normal(g, (T, sum(slices)), 1.0, dtype)
    offs = [sum(slices[:i]) for i in range(S)]
    return Case(f"decode_qkv_T{T}", dtype, x, A, B, out, offs, r, S, L, token_idx=idx,
                scale=1.0, add=True, meta={"T": T})


def prefill_seg_lens(g, n_req: int = 8, lo: int = 8, hi: int = 2048) -> List[int]:
    u = torch.rand(n_req, generator=g, dtype=torch.float64)
    return [int(round(math.exp(math.log(lo) + float(v) * (math.log(hi) - math.log(lo)))))
            for v in u]


def prefill_gateup(r: int = 16, seed: Optional[int] = None, H: int = 4096, N: int = GATEUP_N,
                   dtype=torch.float16, seg_loras=(0, 0, 0, 1, 2, 2, 3, 3),
                   lens: Optional[List[int]] = None) -> Case:
    g = _gen(SEED_BASE + 3 if seed is None else seed)
    if lens is None:
        lens = prefill_seg_lens(g, len(seg_loras))
    L = max(seg_loras) + 1
    T = sum(lens)
    starts = [sum(lens[:i]) for i in range(len(lens))]
    x = _normal(g, (T, H), 1.0, dtype)
    A = _normal(g, (L, 2 * r, H), WEIGHT_STD, dtype)
    B = [_normal(g, (L, N, r), WEIGHT_STD, dtype) for _ in range(2)]
    out = _normal(g, (T, 2 * N), 1.0, dtype)
    i32 = torch.int32
    return Case(f"prefill_gateup_r{r}", dtype, x, A, B, out, [0, N], r, 2, L,
                seg_start=torch.tensor(starts, dtype=i32),
                seg_len=torch.tensor(lens, dtype=i32),
                seg_lora=torch.tensor(list(seg_loras), dtype=i32),
                scale=1.0, add=True, meta={"lens": lens, "T": T})


def zipf_ids(g, T: int, L: int, s: float = 1.1) -> torch.Tensor:
    w = torch.tensor([(l + 1) ** (-s) for l in range(L)], dtype=torch.float64)
    return torch.multinomial(w / w.sum(), T, replacement=True, generator=g).to(torch.int32)


def mixed_rank_70b(N: int = 8192, seed: Optional[int] = None, T: int = 2048, H: int = 8192,
                   L: int = 32, dtype=torch.bfloat16, sgmv: bool = False,
                   pad_fill: str = "garbage", inactive: float = 0.05) -> Case:
    """Rows/columns beyond an adapter's rank hold ``pad_fill`` ('garbage' = random
    values a rank-aware kernel must never read into the result, 'zero' = the
    zero padding a max-rank kernel multiplies through)."""
    g = _gen(SEED_BASE + 4 if seed is None else seed)
    choices = torch.tensor(MIXED_RANKS, dtype=torch.int32)
    ranks = choices[torch.randint(0, len(MIXED_RANKS), (L,), generator=g)]
    R = int(ranks.max())
    x = _normal(g, (T, H), 1.0, dtype)
    A = _normal(g, (L, R, H), WEIGHT_STD, dtype)
    B = _normal(g, (L, N, R), WEIGHT_STD, dtype)
    fill = 0.0 if pad_fill == "zero" else None
    for l in range(L):
        rl = int(ranks[l])
        if fill is not None:
            A[l, rl:, :] = 0
            B[l, :, rl:] = 0
    ids = zipf_ids(g, T, L)
    ids[_exact_inactive(g, T, inactive)] = -1
    out = _normal(g, (T, N), 1.0, dtype)
    case = Case(f"mixed_rank_70b_N{N}", dtype, x, A, [B], out, [0], R, 1, L,
                ranks=ranks.clone(), scale=1.0, add=True, meta={"N": N})
    if sgmv:
        order = torch.argsort(ids.to(torch.int64), stable=True)
        case.x = x[order].contiguous()
        case.out = out[order].contiguous()
        sid = ids[order]
        case.seg_start, case.seg_len, case.seg_lora = _segments_from_sorted(sid)
        case.name += "_sgmv"
    else:
        case.token_idx = ids
    return case


def mixed_rank_map(T: int = 2048, L: int = 32, seed: Optional[int] = None,
                   inactive: float = 0.05, sgmv: bool = False):
    """The token -> adapter structure of the mixed-rank workload without its
    tensors (for timing runs that draw the tensors on the device): ranks [L]
    uniform over MIXED_RANKS, Zipf(1.1) adapter per token with exactly
    round(inactive * T) tokens at -1.  Same recipe as ``mixed_rank_70b``, own
    random stream.  Returns (ranks, token_idx) or, with sgmv, (ranks,
    (seg_start, seg_len, seg_lora)) over the tokens sorted by adapter."""
    g = _gen(SEED_BASE + 40 if seed is None else seed)
    choices = torch.tensor(MIXED_RANKS, dtype=torch.int32)
    ranks = choices[torch.randint(0, len(MIXED_RANKS), (L,), generator=g)]
    ids = zipf_ids(g, T, L)
    ids[_exact_inactive(g, T, inactive)] = -1
    if not sgmv:
        return ranks, ids
    sid, _ = torch.sort(ids.to(torch.int64), stable=True)
    return ranks, _segments_from_sorted(sid.to(torch.int32))


def sweep(H: int, batch: int, seq_len: int, seed: Optional[int] = None, r: int = 16,
          L: int = 4, dtype=torch.float16, which: str = "both") -> Case:
    """One point of the microbenchmark sweep: N = H, add_inputs=True, sorted ids."""
    if seed is None:
        seed = SEED_BASE + 5 + 1000 * SWEEP_H.index(H) if H in SWEEP_H else SEED_BASE + 5
        seed += 17 * batch + seq_len
    g = _gen(seed)
    T = batch * seq_len
    x = _normal(g, (T, H), 1.0, dtype)
    A = _normal(g, (L, r, H), WEIGHT_STD, dtype)
    B = _normal(g, (L, H, r), WEIGHT_STD, dtype)
    out = _normal(g, (T, H), 1.0, dtype)
    req_ids, _ = torch.sort(torch.randint(0, L, (batch,), generator=g, dtype=torch.int32))
    case = Case(f"sweep_H{H}_b{batch}_sl{seq_len}", dtype, x, A, [B], out, [0], r, 1, L,
                scale=1.0, add=True, meta={"H": H, "batch": batch, "seq_len": seq_len})
    if seq_len == 1:
        case.token_idx = req_ids.clone()
    else:
        i32 = torch.int32
        case.seg_start = torch.arange(batch, dtype=i32) * seq_len
        case.seg_len = torch.full((batch,), seq_len, dtype=i32)
        case.seg_lora = req_ids.clone()
    return case


def pages_point(seed: Optional[int] = None, dtype=torch.float16) -> Case:
    """The printed microbenchmark point: 16 requests x 16 tokens (m = 256),
    r = 16, n = 2048, 4 adapters, sorted request ids, add_inputs=False.  The
    shrink side (not part of the printed point) uses H = n."""
    case = sweep(H=2048, batch=16, seq_len=16, seed=SEED_BASE + 6 if seed is None else seed,
                 dtype=dtype)
    case.name = "pages_point_m256_r16_n2048"
    case.add = False
    case.meta = {"m": 256, "batch": 16, "seq_len": 16, "n": 2048}
    return case


def model_shape(name: str, T: int, seed: Optional[int] = None, r: int = 16, L: int = 4,
                dtype=torch.bfloat16) -> Case:
    """A decode batch (as ``decode_qkv``: 10 % of tokens idx=-1, the rest
    uniform over L adapters) for one Llama-3 o_proj / down_proj shape."""
    H, N = MODEL_SHAPES[name]
    if seed is None:
        seed = SEED_BASE + 7 + 100 * list(MODEL_SHAPES).index(name) + T
    case = decode_qkv(T, seed=seed, H=H, r=r, L=L, slices=(N,), dtype=dtype)
    case.name = f"{name}_T{T}"
    case.meta = {"T": T, "H": H, "N": N}
    return case
