"""Shrink / expand / expand_slice on the GPU against the oracle, element by
element, on the seeded workloads and on edge cases."""
import numpy as np
import pytest
import torch

import oracle
import lora_inputs as li
from helpers import (assert_close, assert_expand_ulp, assert_y_fp32, f64, gpu_plan, gpu_run,
                     oracle_map, oracle_run)

pytestmark = pytest.mark.gpu


def full_check(lg, case, rows=None):
    """End to end against the oracle (the output type's tolerance), then y
    within the fp32-accumulation bound and out within one ulp of the
    oracle's expand of the GPU's own y."""
    y, out, plan = gpu_run(lg, case)
    y_ref, o_ref = oracle_run(case, rows)
    assert_y_fp32(y, case, rows, case.name)
    assert_expand_ulp(out, y, case, rows, case.name)
    if rows is not None:
        y, out = y[rows], out[rows]
    assert_close(out, o_ref, case.dtype, f"{case.name} out")
    return y, out, plan


# ---------------------------------------------------------------- workloads

def test_bgmv_small(cuda_lib):
    c = li.bgmv_small()
    y, out, _ = full_check(cuda_lib, c)
    # inactive tokens: y rows zero, out rows untouched bit for bit
    m = (c.token_idx == -1).numpy()
    assert (y.numpy()[m] == 0).all()
    assert torch.equal(out[m].view(torch.int16), c.out[m].view(torch.int16))


@pytest.mark.parametrize("T", li.DECODE_T)
def test_decode_qkv(cuda_lib, T):
    c = li.decode_qkv(T)
    y, out, _ = full_check(cuda_lib, c)
    m = (c.token_idx == -1).numpy()
    assert torch.equal(out[m].view(torch.int16), c.out[m].view(torch.int16))


@pytest.mark.parametrize("T", li.DECODE_T)
def test_decode_qkv_no_add(cuda_lib, T):
    """add_inputs=False: out is the LoRA term alone, so the tolerance applies
    to it directly (bf16, the warp-streaming expand)."""
    c = li.decode_qkv(T)
    c.add = False
    y, out, _ = full_check(cuda_lib, c)
    m = (c.token_idx == -1).numpy()
    assert (out[m].float() == 0).all()


@pytest.mark.parametrize("r", (16, 32, 64))
def test_prefill_gateup_no_add(cuda_lib, r):
    c = li.prefill_gateup(r=r)
    c.add = False
    rows = np.sort(np.random.default_rng(r + 1).choice(c.T, size=min(c.T, 384), replace=False))
    full_check(cuda_lib, c, rows)


@pytest.mark.parametrize("N,sgmv", [(8192, False), (28672, False), (8192, True)])
def test_mixed_rank_70b_no_add(cuda_lib, N, sgmv):
    c = li.mixed_rank_70b(N=N, sgmv=sgmv)
    c.add = False
    rows = np.sort(np.random.default_rng(N + 1).choice(c.T, size=256, replace=False))
    full_check(cuda_lib, c, rows)


@pytest.mark.parametrize("r", (16, 32, 64))
def test_prefill_gateup(cuda_lib, r):
    c = li.prefill_gateup(r=r)
    g = np.random.default_rng(r)
    rows = np.sort(g.choice(c.T, size=min(c.T, 384), replace=False))
    full_check(cuda_lib, c, rows)


@pytest.mark.parametrize("N,sgmv", [(8192, False), (28672, False), (8192, True)])
def test_mixed_rank_70b(cuda_lib, N, sgmv):
    c = li.mixed_rank_70b(N=N, sgmv=sgmv)
    g = np.random.default_rng(N)
    rows = np.sort(g.choice(c.T, size=256, replace=False))
    full_check(cuda_lib, c, rows)


@pytest.mark.parametrize("H", li.SWEEP_H)
@pytest.mark.parametrize("batch,sl", [(16, 1), (512, 1), (16, 8), (2048, 8)])
def test_sweep_points(cuda_lib, H, batch, sl):
    c = li.sweep(H=H, batch=batch, seq_len=sl)
    rows = None
    if c.T > 512:
        rows = np.sort(np.random.default_rng(H + batch).choice(c.T, 512, replace=False))
    full_check(cuda_lib, c, rows)


def test_pages_point(cuda_lib):
    """The microbenchmark PR's printed SGMV expand point (m = 256 as 16 x 16,
    r = 16, n = 2048, 4 sorted adapters, add_inputs=False), and the same
    shape with one adapter over one segment (the dense special case)."""
    c = li.pages_point()
    full_check(cuda_lib, c)
    c.seg_start = torch.zeros(1, dtype=torch.int32)
    c.seg_len = torch.full((1,), c.T, dtype=torch.int32)
    c.seg_lora = torch.zeros(1, dtype=torch.int32)
    full_check(cuda_lib, c)


@pytest.mark.parametrize("name", list(li.MODEL_SHAPES))
@pytest.mark.parametrize("T", [200, 1024])
def test_model_shapes(cuda_lib, name, T):
    """Llama-3 o_proj / down_proj shapes (H up to 28672) at decode batches."""
    c = li.model_shape(name, T)
    rows = None if T <= 200 else np.sort(np.random.default_rng(T).choice(c.T, 192, replace=False))
    full_check(cuda_lib, c, rows)


def test_sweep_largest_point_sampled(cuda_lib):
    """batch 8192 x seq-len 8 = 65536 tokens at H = N = 16384: sampled rows."""
    c = li.sweep(H=16384, batch=8192, seq_len=8)
    rows = np.sort(np.random.default_rng(0).choice(c.T, 96, replace=False))
    full_check(cuda_lib, c, rows)


# ---------------------------------------------------------------- invariants

def test_bgmv_equals_sgmv_bitwise(cuda_lib):
    """Punica issue #17: BGMV semantics are a subset of SGMV's.  The same
    token -> adapter map given both ways gives bit-identical results."""
    lg = cuda_lib
    c = li.prefill_gateup(r=16, H=1024, N=1000, lens=[70, 5, 130, 64, 1, 9, 200, 33])
    y_s, o_s, _ = gpu_run(lg, c)
    c.token_idx = c.lora_of_token()
    y_b, o_b, _ = gpu_run(lg, c)
    assert torch.equal(y_s, y_b)
    assert torch.equal(o_s.view(torch.int16), o_b.view(torch.int16))


def test_expand_slice_equals_back_to_back(cuda_lib):
    lg = cuda_lib
    c = li.decode_qkv(200, seed=77)
    plan = gpu_plan(lg, c, "cuda")
    y = torch.randn(c.T, 48, generator=torch.Generator().manual_seed(1)).cuda()
    Bs = [b.cuda() for b in c.B]
    o1 = c.out.cuda()
    lg.lora_expand_slice(y, Bs, o1, plan, c.slice_offsets, y_slice_stride=16)
    o2 = c.out.cuda()
    for s in range(3):
        lg.lora_expand_slice(y, [Bs[s]], o2, plan, [c.slice_offsets[s]], y_slice_stride=0,
                             ) if s == 0 else lg.lora_expand_slice(
            y[:, 16 * s:], [Bs[s]], o2, plan, [c.slice_offsets[s]], y_slice_stride=0)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_rank_aware_equals_padded(cuda_lib):
    """Punica issue #17: zero-padding ranks up to the largest changes nothing."""
    lg = cuda_lib
    kw = dict(T=300, H=512, L=8, N=384)
    cg = li.mixed_rank_70b(pad_fill="garbage", **kw)
    cz = li.mixed_rank_70b(pad_fill="zero", **kw)
    y_g, o_g, _ = gpu_run(lg, cg)
    cz.ranks = None
    y_z, o_z, _ = gpu_run(lg, cz)
    assert_close(o_g, f64(o_z), cg.dtype, "out")
    # and both against the oracle
    _, o_ref = oracle_run(cg)
    assert_y_fp32(y_g, cg, what="rank-aware")
    assert_y_fp32(y_z, cg, what="padded")
    assert_expand_ulp(o_g, y_g, cg, what="rank-aware")
    assert_close(o_g, o_ref, cg.dtype, "out vs oracle")


def test_single_adapter_equals_dense(cuda_lib):
    """One adapter, every token: shrink = x A^T, expand = out + y B^T (the
    torch.mm single-LoRA roofline of vLLM PR #11579), checked against a plain
    fp64 matmul."""
    lg = cuda_lib
    g = torch.Generator().manual_seed(5)
    T, H, R, N = 333, 1536, 16, 2048
    x = torch.randn(T, H, generator=g).half()
    A = (torch.randn(1, R, H, generator=g) * 0.02).half()
    B = (torch.randn(1, N, R, generator=g) * 0.02).half()
    out0 = torch.randn(T, N, generator=g).half()
    plan = lg.new_plan(T, 1)
    lg.lora_group_tokens(torch.zeros(T, dtype=torch.int32).cuda(), 1, plan)
    y = torch.empty(T, R, device="cuda")
    lg.lora_shrink(x.cuda(), A.cuda(), y, plan)
    out = out0.cuda()
    lg.lora_expand(y, B.cuda(), out, plan, add_inputs=True)
    torch.cuda.synchronize()
    y_ref = f64(x) @ f64(A[0]).T
    mag = np.abs(f64(x)) @ np.abs(f64(A[0])).T
    assert (np.abs(f64(y) - y_ref) <= 1e-5 * mag + 1e-7).all()   # the fp32 bound of helpers
    assert_close(out, f64(out0) + y_ref @ f64(B[0]).T, torch.float16, "out")
    o_own = f64(out0) + f64(y) @ f64(B[0]).T      # the expand of the GPU's own y
    from helpers import ulp
    bound = ulp(np.maximum(np.abs(f64(out)), np.abs(o_own)), torch.float16) \
        + 2.0 ** -14 * (np.abs(f64(y)) @ np.abs(f64(B[0])).T)
    assert (np.abs(f64(out) - o_own) <= bound).all()


@pytest.mark.parametrize("R,ranks", [(16, None), (64, None), (32, [32, 20])])
@pytest.mark.parametrize("add", [False, True])
def test_segments_interleaving_adapters(cuda_lib, R, ranks, add):
    """SGMV segments not sorted by adapter (64 one-token segments alternating
    over 2 adapters, then longer alternating runs): every segment becomes its
    own group and tile, far more tiles than the T/64 + L + 1 bound that
    covers BGMV plans.  Both the warp-streaming (r = 16) and the tensor-core
    (r = 64, and r = 32 on a large batch) expand must reach every tile."""
    T = 64 + 8 * 120 + (2048 if R == 32 else 0)
    c = make_case(T, 256, R, 2, [512, 256], torch.float16, seed=R + add, add=add, ranks=ranks)
    starts, lens, loras = [], [], []
    t = 0
    for i in range(64):                       # one-token segments A B A B ...
        starts.append(t); lens.append(1); loras.append(i % 2); t += 1
    while t < T:                              # then runs of 7 to 120 tokens, alternating
        n = min(T - t, 7 + (len(starts) * 37) % 114)
        starts.append(t); lens.append(n); loras.append(len(starts) % 2); t += n
    c.token_idx = None
    c.seg_start = torch.tensor(starts, dtype=torch.int32)
    c.seg_len = torch.tensor(lens, dtype=torch.int32)
    c.seg_lora = torch.tensor(loras, dtype=torch.int32)
    y, out, plan = full_check(cuda_lib, c)
    ntiles = int(cuda_lib.plan_view(plan, c.T, c.L)["header"][cuda_lib.HDR["NTILES"]])
    assert ntiles > (T + 63) // 64 + 2 + 1


@pytest.mark.parametrize("R,ranks,Ns", [(24, [24, 5, 13, 0], [256, 128, 96]),
                                         (64, [64, 40, 17], [512, 256]),
                                         (32, None, [384, 384, 128])])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("add", [False, True])
def test_sorted_segments_rank_aware(cuda_lib, R, ranks, Ns, dtype, add):
    """Long sorted segments (tiles of consecutive token rows, copied by TMA
    in the tensor-core shrink) with ranks below R, several slices and an H
    that is not a multiple of the 128-wide stage."""
    L = len(ranks) if ranks is not None else 3
    T = 700
    c = make_case(T, 640, R, L, Ns, dtype, seed=R + L + add, add=add, ranks=ranks)
    lens = [200, 90, 250, T - 540]
    c.token_idx = None
    c.seg_start = torch.tensor(np.cumsum([0] + lens[:-1]), dtype=torch.int32)
    c.seg_len = torch.tensor(lens, dtype=torch.int32)
    c.seg_lora = torch.tensor([0, 0, 1, L - 1], dtype=torch.int32)  # sorted: a run of adapter 0
    full_check(cuda_lib, c)


@pytest.mark.parametrize("T,R,Ns,lens", [
    (256, 64, [200, 72], [128, 128]),              # full tiles, ragged last chunks
    (320, 128, [384, 136], [64, 192, 64]),         # R = 128: two TMA B boxes per chunk
    (2048, 16, [2048, 200], [700, 600, 748]),      # rank 16 on the tensor-core expand
    (131, 64, [256], [131]),                       # a partial tile ending at T
])
@pytest.mark.parametrize("add", [True, False])
def test_sorted_segments_tma_expand(cuda_lib, T, R, Ns, lens, add):
    """Tiles of consecutive rows through the tensor-core expand: out blocks
    loaded (and, for full tiles and full chunks, stored) by TMA, B by TMA at
    full rank; ragged chunks and partial tiles keep plain stores."""
    L = len(lens)
    c = make_case(T, 256, R, L, Ns, torch.bfloat16, seed=T + R + add, add=add)
    c.token_idx = None
    c.seg_start = torch.tensor(np.cumsum([0] + lens[:-1]), dtype=torch.int32)
    c.seg_len = torch.tensor(lens, dtype=torch.int32)
    c.seg_lora = torch.arange(L, dtype=torch.int32)
    full_check(cuda_lib, c)


# ---------------------------------------------------------------- edge cases

def make_case(T, H, R, L, N_list, dtype, seed, *, S=None, p_neg=0.2, add=True, scale=0.7,
              sscale=1.3, ranks=None, offsets=None, N_total=None):
    g = torch.Generator().manual_seed(seed)
    S = S if S is not None else len(N_list)
    x = torch.randn(T, H, generator=g).to(dtype)
    A = (torch.randn(L, S * R, H, generator=g) * 0.05).to(dtype)
    B = [(torch.randn(L, n, R, generator=g) * 0.05).to(dtype) for n in N_list]
    if offsets is None:
        offsets = [sum(N_list[:i]) for i in range(len(N_list))]
    N_total = N_total or (max(o + n for o, n in zip(offsets, N_list)) if N_list else 0)
    out = torch.randn(T, N_total, generator=g).to(dtype)
    idx = torch.randint(0, L, (T,), generator=g, dtype=torch.int32)
    neg = torch.rand(T, generator=g) < p_neg
    idx[neg] = -1
    c = li.Case(f"edge_T{T}_H{H}_R{R}_L{L}", dtype, x, A, B, out, offsets, R, S, L,
                token_idx=idx, scale=scale, add=add)
    c.shrink_scale = sscale
    if ranks is not None:
        c.ranks = torch.tensor(ranks, dtype=torch.int32)
    return c


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("T,H,R,L,Ns", [
    (1, 64, 16, 1, [64]),          # single token
    (65, 1000, 16, 3, [200]),      # ragged tile, H not a multiple of 64
    (130, 2049, 16, 4, [2049]),    # odd H and odd N: scalar paths
    (77, 7, 3, 2, [5]),            # tiny odd everything
    (129, 4096, 1, 2, [128]),      # rank 1
    (64, 4096, 20, 5, [1032]),     # rank 20 (not a bin of 16)
    (100, 640, 128, 3, [384]),     # rank 128, MMA over 8 k-steps
    (300, 512, 48, 2, [256, 100]), # 2 slices (3 y blocks would exceed)
])
def test_edge_shapes(cuda_lib, dtype, T, H, R, L, Ns):
    c = make_case(T, H, R, L, Ns, dtype, seed=T * 7 + H)
    full_check(cuda_lib, c)


# Ranks above 48 take the tcgen05 expand: rank-aware adapters (ranks 0, 1,
# 17, 33 and the full R, K steps padded past the rank), R not a multiple of
# 16, both add_inputs settings, ragged tiles and slices.
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("add", [False, True])
@pytest.mark.parametrize("T,R,ranks,Ns", [
    (200, 64, [0, 1, 17, 33, 64], [256, 136]),
    (77, 56, None, [200]),
    (130, 128, [128, 65, 3], [384, 8]),
])
def test_large_rank_expand(cuda_lib, dtype, add, T, R, ranks, Ns):
    L = len(ranks) if ranks else 3
    c = make_case(T, 512, R, L, Ns, dtype, seed=T + R + add, add=add, ranks=ranks)
    full_check(cuda_lib, c)


# Large batches give each tensor-core expand CTA a span of several 128-column
# chunks (pipelined out / B blocks, y converted once); ranks 17-48 take that
# kernel too once spans hold two or more chunks.  Ragged last chunks (slices
# of 2600 and 2504 columns), rank-0 adapters and -1 tokens, both dtypes and
# add_inputs settings; sampled rows, and every inactive row checked in full.
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("add", [False, True])
@pytest.mark.parametrize("R,ranks", [(32, [32, 9, 0, 20]), (64, [64, 0, 17, 33, 40]),
                                     (100, [100, 65, 0, 3])])
def test_tensor_expand_spans(cuda_lib, dtype, add, R, ranks):
    c = make_case(4096, 256, R, len(ranks), [2600, 2504], dtype, seed=R + 3 * add, add=add,
                  ranks=ranks)
    rows = np.sort(np.random.default_rng(R).choice(c.T, 256, replace=False))
    y, out_full, _ = gpu_run(cuda_lib, c)
    y_ref, o_ref = oracle_run(c, rows)
    assert_y_fp32(y, c, rows, c.name)
    assert_expand_ulp(out_full, y, c, rows, c.name)
    assert_close(out_full[rows], o_ref, c.dtype, f"{c.name} out")
    idx = c.token_idx.numpy()
    inactive = (idx == -1) | (c.ranks.numpy()[np.maximum(idx, 0)] == 0)
    if add:
        assert torch.equal(out_full[inactive].view(torch.int16), c.out[inactive].view(torch.int16))
    else:
        assert (out_full[inactive].float() == 0).all()


def skewed_idx(T, counts, seed):
    """Token indices giving adapter a exactly counts[a] tokens (the rest -1),
    shuffled: tiles of every size in one batch."""
    idx = torch.full((T,), -1, dtype=torch.int32)
    pos = torch.randperm(T, generator=torch.Generator().manual_seed(seed))
    k = 0
    for a, n in enumerate(counts):
        idx[pos[k:k + n]] = a
        k += n
    return idx


# The shrink's warps split a tile's k steps when the batch averages at most 16
# tokens per adapter, else its n-tiles; both must hold for tiles of every size
# (1..64 tokens) and every A-row count (1..16 n-tiles).
@pytest.mark.parametrize("T,L,counts", [
    (64, 4, [60, 1, 2, 0]),           # k-split warps, one near-full tile
    (48, 4, [33, 9, 0, 5]),           # k-split warps, 3 row blocks
    (200, 4, [150, 1, 20, 3]),        # n-split warps, 1- and 3-token tiles
    (1024, 8, [900, 1, 2, 4, 17, 31, 40, 29]),
])
@pytest.mark.parametrize("R,S", [(16, 3), (64, 2), (8, 1), (20, 1)])
def test_warp_splits_every_tile_size(cuda_lib, T, L, counts, R, S):
    c = make_case(T, 512, R, L, [96] * S, torch.bfloat16, seed=T + R + S, sscale=1.0)
    c.token_idx = skewed_idx(T, counts, seed=T + L)
    full_check(cuda_lib, c)


@pytest.mark.parametrize("add", [False, True])
def test_add_flag_and_inactive_rows(cuda_lib, add):
    c = make_case(150, 256, 16, 3, [512], torch.float16, seed=3, add=add, p_neg=0.3)
    y, out, _ = full_check(cuda_lib, c)
    m = (c.token_idx == -1).numpy()
    if add:
        assert torch.equal(out[m].view(torch.int16), c.out[m].view(torch.int16))
    else:
        assert (out[m].float() == 0).all()
    assert (y.numpy()[m] == 0).all()


def test_all_tokens_inactive(cuda_lib):
    c = make_case(100, 128, 16, 2, [256], torch.bfloat16, seed=4, p_neg=1.1)
    y, out, _ = full_check(cuda_lib, c)
    assert torch.equal(out.view(torch.int16), c.out.view(torch.int16))


def test_mixed_ranks_with_zero_and_slices(cuda_lib):
    c = make_case(400, 1024, 32, 6, [320, 96, 96], torch.bfloat16, seed=9,
                  ranks=[0, 1, 7, 16, 31, 32])
    full_check(cuda_lib, c)


def test_slices_with_gaps_and_wide_out(cuda_lib):
    """Slices placed at offsets with gaps inside a wider out: gap columns untouched."""
    c = make_case(90, 256, 16, 3, [64, 48], torch.float16, seed=11, offsets=[8, 120],
                  N_total=200, add=False)
    y, out, _ = full_check(cuda_lib, c)
    keep = np.r_[0:8, 72:120, 168:200]
    assert torch.equal(out[:, keep].view(torch.int16), c.out[:, keep].view(torch.int16))


def test_strided_x_y_out(cuda_lib):
    """Leading dimensions larger than the logical widths."""
    lg = cuda_lib
    c = make_case(70, 512, 16, 3, [256], torch.float16, seed=12)
    dev = "cuda"
    plan = gpu_plan(lg, c, dev)
    xb = torch.zeros(c.T, 520, dtype=c.dtype)
    xb[:, :512] = c.x
    xd = xb.to(dev)[:, :512]
    yb = torch.full((c.T, 24), 123.0, device=dev)
    y = yb[:, :16]
    ob = torch.zeros(c.T, 264, dtype=c.dtype)
    ob[:, :256] = c.out
    od = ob.to(dev)
    out = od[:, :256]
    lg.lora_shrink(xd, c.A.to(dev), y, plan, scale=c.shrink_scale)
    lg.lora_expand(y, c.B[0].to(dev), out, plan, scale=c.scale, add_inputs=True)
    torch.cuda.synchronize()
    y_ref, o_ref = oracle_run(c)
    assert_y_fp32(y.cpu(), c, what="strided")
    assert_expand_ulp(out.cpu(), y.cpu(), c, what="strided")
    assert_close(out.cpu(), o_ref, c.dtype, "out")
    assert (yb[:, 16:].cpu() == 123.0).all()
    assert (od[:, 256:].cpu().float() == 0).all()


def test_shrink_add_inputs_accumulates(cuda_lib):
    lg = cuda_lib
    c = make_case(80, 384, 16, 2, [64], torch.float16, seed=13)
    plan = gpu_plan(lg, c, "cuda")
    y0 = torch.randn(c.T, 16, generator=torch.Generator().manual_seed(2))
    y = y0.cuda()
    lg.lora_shrink(c.x.cuda(), c.A.cuda(), y, plan, scale=0.5, add_inputs=True)
    torch.cuda.synchronize()
    lo, _, _ = oracle_map(c)
    ref = oracle.shrink(f64(c.x), f64(c.A), lo, scale=0.5, add=True, y=y0.double().numpy())
    mag = oracle.shrink(np.abs(f64(c.x)), np.abs(f64(c.A)), lo, scale=0.5) + np.abs(f64(y0))
    assert (np.abs(f64(y) - ref) <= 1e-5 * mag + 1e-7).all()   # the fp32 bound of helpers


def test_plan_mismatch_writes_nothing(cuda_lib):
    lg = cuda_lib
    c = make_case(50, 128, 16, 3, [64], torch.float16, seed=14)
    plan = lg.new_plan(c.T, c.L)
    lg.lora_group_tokens(c.token_idx.cuda(), c.L, plan)
    # an operator told a different L than the plan was built with
    y = torch.full((c.T, 16), 7.0, device="cuda")
    lg.lora_shrink(c.x.cuda(), torch.cat([c.A, c.A]).cuda(), y, plan)
    torch.cuda.synchronize()
    assert (y.cpu() == 7.0).all()
    bad, err = lg.lora_get_error(plan)
    assert err & lg.PLANERR_MISMATCH


def test_empty_batch_is_noop(cuda_lib):
    lg = cuda_lib
    plan = lg.new_plan(0, 2)
    lg.lora_group_tokens(torch.empty(0, dtype=torch.int32, device="cuda"), 2, plan)
    x = torch.empty(0, 64, dtype=torch.float16, device="cuda")
    y = torch.empty(0, 16, device="cuda")
    lg.lora_shrink(x, torch.zeros(2, 16, 64, dtype=torch.float16, device="cuda"), y, plan)
    lg.lora_expand(y, torch.zeros(2, 32, 16, dtype=torch.float16, device="cuda"),
                   torch.empty(0, 32, dtype=torch.float16, device="cuda"), plan)
    torch.cuda.synchronize()


def test_rejects_bad_arguments(cuda_lib):
    lg = cuda_lib
    c = make_case(10, 64, 16, 2, [32], torch.float16, seed=15)
    plan = gpu_plan(lg, c, "cuda")
    y = torch.zeros(10, 16, device="cuda")
    out = c.out.cuda()
    B = c.B[0].cuda()
    with pytest.raises(lg.LoraError):  # overlapping slices
        lg.lora_expand_slice(y, [B, B], torch.zeros(10, 64, dtype=torch.float16, device="cuda"),
                             plan, [0, 16], y_slice_stride=0)
    with pytest.raises(lg.LoraError):  # rank above 128
        lg.lora_expand(torch.zeros(10, 130, device="cuda"),
                       torch.zeros(2, 32, 130, dtype=torch.float16, device="cuda"), out, plan)
    with pytest.raises(lg.LoraError):  # plan too small
        lg.lora_group_tokens(c.token_idx.cuda(), 2, plan[:64])
    with pytest.raises(ValueError):  # CPU tensor: no CPU path
        lg.lora_expand(y.cpu(), B, out, plan)
