"""The plan-free BGMV operators (lora_bgmv_shrink, lora_bgmv_expand_slice,
lora_bgmv_shrink_expand_slice) against the oracle, element by element.

Every shape runs both as the chained pair and as the two separate calls.
Bounds are those of helpers.py: y within the fp32-accumulation bound, out
within one ulp of the oracle's expand of the GPU's own y, and out end to end
within the output type's tolerance."""
import numpy as np
import pytest
import torch

import lora_inputs as li
from helpers import assert_close, assert_expand_ulp, assert_y_fp32, f64, gpu_run, oracle_run
from test_gpu_ops import make_case, skewed_idx

pytestmark = pytest.mark.gpu


def bgmv_run(lg, case, chained=True, dev="cuda", y_fill=float("nan"), status=None):
    """The plan-free path on the GPU.  Returns (y, out) on the host."""
    x, A = case.x.to(dev), case.A.to(dev)
    Bs = [b.to(dev) for b in case.B]
    out = case.out.to(dev)
    idx = case.token_idx.to(dev) if case.token_idx is not None else None
    ranks = case.ranks.to(dev) if case.ranks is not None else None
    y = torch.full((case.T, case.num_slices * case.R), y_fill, dtype=torch.float32, device=dev)
    if chained:
        lg.lora_bgmv_shrink_expand_slice(x, A, y, Bs, out, case.slice_offsets, idx, ranks=ranks,
                                         scale_shrink=case.shrink_scale, scale_expand=case.scale,
                                         add_inputs=case.add, status=status)
    else:
        lg.lora_bgmv_shrink(x, A, y, idx, num_slices=case.num_slices, ranks=ranks,
                            scale=case.shrink_scale, status=status)
        lg.lora_bgmv_expand_slice(y, Bs, out, case.slice_offsets, idx, y_slice_stride=case.R,
                                  ranks=ranks, scale=case.scale, add_inputs=case.add,
                                  status=status)
    torch.cuda.synchronize()
    return y.cpu(), out.cpu()


def check(lg, case, rows=None, chained=True):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y, out = bgmv_run(lg, case, chained, status=status)
    assert int(status.item()) == 0
    y_ref, o_ref = oracle_run(case, rows)
    assert_y_fp32(y, case, rows, f"{case.name} bgmv")
    assert_expand_ulp(out, y, case, rows, f"{case.name} bgmv")
    if rows is not None:
        y, out = y[rows], out[rows]
    assert_close(out, o_ref, case.dtype, f"{case.name} bgmv out")
    return y, out


def inactive_rows_ok(case, y, out):
    idx = case.token_idx.numpy() if case.token_idx is not None else np.zeros(case.T, np.int32)
    m = (idx < 0) | (idx >= case.L)
    if case.ranks is not None:
        m |= case.ranks.numpy()[np.clip(idx, 0, case.L - 1)] <= 0
    assert (y.numpy()[(idx < 0) | (idx >= case.L)] == 0).all()
    if case.add:
        assert torch.equal(out[m].view(torch.int16), case.out[m].view(torch.int16))
    else:
        assert (out[m].float() == 0).all()


# ---------------------------------------------------------------- workloads

@pytest.mark.parametrize("T", li.DECODE_T + (333, 700, 2000))
@pytest.mark.parametrize("add", [True, False])
@pytest.mark.parametrize("chained", [True, False])
def test_decode_qkv(cuda_lib, T, add, chained):
    """The decode q/k/v batches, plus batch sizes whose per-CTA work ranges
    of the persistent expand cross slice and token-block boundaries."""
    c = li.decode_qkv(T) if T in li.DECODE_T else li.decode_qkv(T, seed=T)
    c.add = add
    y, out = check(cuda_lib, c, chained=chained)
    inactive_rows_ok(c, y, out)


def test_bgmv_small(cuda_lib):
    c = li.bgmv_small()
    y, out = check(cuda_lib, c)
    inactive_rows_ok(c, y, out)


@pytest.mark.parametrize("name", list(li.MODEL_SHAPES))
@pytest.mark.parametrize("T", [16, 1024])
def test_model_shapes(cuda_lib, name, T):
    """Llama-3 o_proj / down_proj (H up to 28672: long K ranges per CTA)."""
    c = li.model_shape(name, T)
    rows = None if T <= 16 else np.sort(np.random.default_rng(T).choice(c.T, 160, replace=False))
    check(cuda_lib, c, rows)


@pytest.mark.parametrize("H", [1024, 4096, 16384])
@pytest.mark.parametrize("batch", [16, 512, 8192])
def test_sweep_points_seq_len_1(cuda_lib, H, batch):
    """The microbenchmark sweep's BGMV points (seq-len 1, sorted ids, fp16)."""
    c = li.sweep(H=H, batch=batch, seq_len=1)
    rows = None if c.T <= 512 else np.sort(np.random.default_rng(H + batch).choice(c.T, 384,
                                                                                    replace=False))
    check(cuda_lib, c, rows)


def test_equals_grouped_path(cuda_lib):
    """The plan-free and the grouped operators compute the same definition."""
    lg = cuda_lib
    c = li.decode_qkv(700, seed=31)
    y_g, o_g, _ = gpu_run(lg, c)
    y_b, o_b = bgmv_run(lg, c)
    assert_close(o_b, f64(o_g), c.dtype, "out bgmv vs grouped")
    mag = np.abs(f64(y_g)) + 1.0
    assert (np.abs(f64(y_b) - f64(y_g)) <= 2e-5 * mag).all()


# ---------------------------------------------------------------- single adapter

def test_single_adapter_no_index(cuda_lib):
    """token_idx = NULL: every token uses adapter 0, no masking (the dense
    single-adapter case; vLLM PR #11579's torch.mm roofline)."""
    lg = cuda_lib
    for T, H, R, N, add in [(256, 2048, 16, 2048, False), (333, 1536, 16, 2048, True),
                            (1, 64, 8, 64, False), (4096, 4096, 64, 4096, True)]:
        c = make_case(T, H, R, 1, [N], torch.float16, seed=T + R, add=add, p_neg=0.0)
        c.token_idx = None
        rows = None if T <= 512 else np.sort(np.random.default_rng(T).choice(T, 256, replace=False))
        check(lg, c, rows)
        # against a plain fp64 matmul as well
        y, out = bgmv_run(lg, c)
        y_ref = c.shrink_scale * (f64(c.x) @ f64(c.A[0]).T)
        o_ref = (f64(c.out) if add else 0) + c.scale * (f64(y) @ f64(c.B[0][0]).T)
        assert_close(out, o_ref, c.dtype, "dense out")
        assert (np.abs(f64(y) - y_ref) <= 1e-5 * (np.abs(f64(c.x)) @ np.abs(f64(c.A[0])).T)
                * abs(c.shrink_scale) + 1e-7).all()


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("T,R,rank,Ns,add", [
    (200, 16, 7, [2048], True),         # rank below R, not a multiple of 4
    (64, 24, 24, [96, 40], False),      # two slices, ragged 64-column chunks
    (300, 32, 0, [512], True),          # rank 0 with add_inputs: out left alone
    (130, 32, 0, [512], False),         # rank 0 without: zeros
    (5000, 8, 8, [1024], True),         # many 64-token tiles
])
def test_single_adapter_ranks_and_slices(cuda_lib, dtype, T, R, rank, Ns, add):
    """The one-adapter expand (no token index) with a rank table, several
    slices and ragged column chunks."""
    c = make_case(T, 512, R, 1, Ns, dtype, seed=T + R + rank, add=add, p_neg=0.0, ranks=[rank])
    c.token_idx = None
    rows = None if T <= 512 else np.sort(np.random.default_rng(T).choice(T, 256, replace=False))
    y, out = check(cuda_lib, c, rows)
    if rank == 0:
        if add:
            assert torch.equal(out.view(torch.int16), (c.out if rows is None else c.out[rows]).view(torch.int16))
        else:
            assert (out.float() == 0).all()


# ---------------------------------------------------------------- edge cases

@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("T,H,R,L,Ns,ranks", [
    (1, 64, 16, 1, [64], None),             # one token, one K stage, no cluster
    (129, 520, 8, 3, [200], None),          # ragged block, H not a multiple of 64, rank 8
    (1000, 256, 16, 8, [96, 96], None),     # 8 adapters, two 64-wide K groups of B_ext
    (77, 1024, 48, 2, [200], [48, 17]),     # rank 48 (3 K steps), a rank below R
    (300, 2048, 16, 5, [256, 104], [16, 0, 7, 16, 1]),  # rank 0 and odd ranks
    (200, 4096, 64, 2, [384, 8], [64, 33]), # rank 64, a slice of 8 columns
    (65, 8192, 8, 8, [136], None),          # long K per CTA, ragged 8-column tail
    (256, 128, 32, 2, [64, 64], None),      # H below one cluster split
    (2000, 1024, 64, 2, [4096], [64, 40]),  # rank 64: tensor-core expand, several items per CTA
    (700, 512, 40, 2, [1024, 128], None),   # rank 40: tensor-core expand, ragged rows
])
@pytest.mark.parametrize("add", [False, True])
def test_edge_shapes(cuda_lib, dtype, T, H, R, L, Ns, ranks, add):
    c = make_case(T, H, R, L, Ns, dtype, seed=T * 3 + H + R, add=add, ranks=ranks)
    y, out = check(cuda_lib, c)
    inactive_rows_ok(c, y, out)


@pytest.mark.parametrize("T,L,counts", [(256, 4, [250, 1, 0, 5]), (1024, 8, [0, 0, 0, 0, 0, 0, 0, 900]),
                                        (130, 3, [0, 130, 0])])
def test_skewed_and_absent_adapters(cuda_lib, T, L, counts):
    """Blocks where some adapters have no token (skipped MMAs and B loads)."""
    c = make_case(T, 1024, 16, L, [384, 128], torch.bfloat16, seed=T + L)
    c.token_idx = skewed_idx(T, counts, seed=T)
    y, out = check(cuda_lib, c)
    inactive_rows_ok(c, y, out)


def test_bad_ids_act_as_no_lora(cuda_lib):
    c = make_case(200, 512, 16, 3, [256], torch.float16, seed=5)
    c.token_idx[::7] = 3
    c.token_idx[::11] = -5
    # the oracle's map treats them as -1 as well
    y, out = check(cuda_lib, c)
    inactive_rows_ok(c, y, out)


@pytest.mark.parametrize("add", [False, True])
def test_all_tokens_inactive(cuda_lib, add):
    c = make_case(300, 256, 16, 2, [256], torch.bfloat16, seed=4, p_neg=1.1, add=add)
    y, out = check(cuda_lib, c)
    inactive_rows_ok(c, y, out)


def test_strided_x_y_out_and_slice_gaps(cuda_lib):
    lg = cuda_lib
    c = make_case(150, 512, 16, 3, [64, 48], torch.float16, seed=12, offsets=[8, 120],
                  N_total=200)
    dev = "cuda"
    xb = torch.zeros(c.T, 520, dtype=c.dtype)
    xb[:, :512] = c.x
    xd = xb.to(dev)[:, :512]
    yb = torch.full((c.T, 40), 123.0, device=dev)
    y = yb[:, :32]
    ob = torch.zeros(c.T, 208, dtype=c.dtype)
    ob[:, :200] = c.out
    od = ob.to(dev)
    out = od[:, :200]
    idx = c.token_idx.to(dev)
    lg.lora_bgmv_shrink(xd, c.A.to(dev), y, idx, num_slices=2, scale=c.shrink_scale)
    lg.lora_bgmv_expand_slice(y, [b.to(dev) for b in c.B], out, c.slice_offsets, idx,
                              y_slice_stride=16, scale=c.scale, add_inputs=True)
    torch.cuda.synchronize()
    _, o_ref = oracle_run(c)
    assert_y_fp32(y.cpu(), c, what="strided")
    assert_expand_ulp(out.cpu(), y.cpu(), c, what="strided")
    assert_close(out.cpu(), o_ref, c.dtype, "strided out")
    assert (yb[:, 32:].cpu() == 123.0).all()
    keep = np.r_[0:8, 72:120, 168:208]
    assert torch.equal(od.cpu()[:, keep].view(torch.int16), ob[:, keep].view(torch.int16))


def test_shrink_add_inputs(cuda_lib):
    lg = cuda_lib
    import oracle
    from helpers import oracle_map
    c = make_case(140, 384, 16, 2, [64], torch.float16, seed=13)
    y0 = torch.randn(c.T, 16, generator=torch.Generator().manual_seed(2))
    y = y0.cuda()
    lg.lora_bgmv_shrink(c.x.cuda(), c.A.cuda(), y, c.token_idx.cuda(), scale=0.5,
                        add_inputs=True)
    torch.cuda.synchronize()
    lo, _, _ = oracle_map(c)
    ref = oracle.shrink(f64(c.x), f64(c.A), lo, scale=0.5, add=True, y=y0.double().numpy())
    mag = oracle.shrink(np.abs(f64(c.x)), np.abs(f64(c.A)), lo, scale=0.5) + np.abs(f64(y0))
    assert (np.abs(f64(y) - ref) <= 1e-5 * mag + 1e-7).all()


def test_empty_batch_and_unsupported_shapes(cuda_lib):
    lg = cuda_lib
    dev = "cuda"
    lg.lora_bgmv_shrink(torch.empty(0, 64, dtype=torch.float16, device=dev),
                        torch.zeros(2, 16, 64, dtype=torch.float16, device=dev),
                        torch.empty(0, 16, device=dev), torch.empty(0, dtype=torch.int32,
                                                                     device=dev))
    c = make_case(10, 64, 16, 9, [32], torch.float16, seed=15)
    y = torch.zeros(10, 16, device=dev)
    with pytest.raises(lg.LoraError) as e:  # more adapters than the plan-free path takes
        lg.lora_bgmv_shrink(c.x.cuda(), c.A.cuda(), y, c.token_idx.cuda())
    assert e.value.status == 2
    c = make_case(10, 60, 16, 2, [32], torch.float16, seed=16)
    with pytest.raises(lg.LoraError) as e:  # H not a multiple of 8
        lg.lora_bgmv_shrink(c.x.cuda(), c.A.cuda(), y, c.token_idx.cuda())
    assert e.value.status == 2
    c = make_case(10, 64, 128, 2, [32], torch.float16, seed=17)
    with pytest.raises(lg.LoraError) as e:  # rank above 64 for the expand
        lg.lora_bgmv_expand_slice(torch.zeros(10, 128, device=dev), [c.B[0].cuda()],
                                  c.out.cuda(), [0], c.token_idx.cuda(), y_slice_stride=0)
    assert e.value.status == 2
