"""lora_shrink_expand_slice (shrink and expand chained by programmatic
dependent launch) against the oracle.

The entry point must give the results of lora_shrink followed by
lora_expand_slice: y in full (fp32) and out, on every workload."""
import numpy as np
import pytest
import torch

import lora_inputs as li
from helpers import (assert_close, assert_expand_ulp, assert_y_fp32, gpu_run, gpu_run_chained,
                     oracle_run)
from test_gpu_ops import make_case

pytestmark = pytest.mark.gpu


def check(lg, case, rows=None):
    y, out, _ = gpu_run_chained(lg, case)
    y_ref, o_ref = oracle_run(case, rows)
    assert_y_fp32(y, case, rows, f"{case.name} chained")
    assert_expand_ulp(out, y, case, rows, f"{case.name} chained")
    if rows is not None:
        y, out = y[rows], out[rows]
    assert_close(out, o_ref, case.dtype, f"{case.name} chained out")
    return y, out


def test_bgmv_small(cuda_lib):
    c = li.bgmv_small()
    y, out = check(cuda_lib, c)
    m = (c.token_idx == -1).numpy()
    assert (y.numpy()[m] == 0).all()
    assert torch.equal(out[m].view(torch.int16), c.out[m].view(torch.int16))


@pytest.mark.parametrize("T", li.DECODE_T)
@pytest.mark.parametrize("add", [True, False])
def test_decode_qkv(cuda_lib, T, add):
    c = li.decode_qkv(T)
    c.add = add
    y, out = check(cuda_lib, c)
    m = (c.token_idx == -1).numpy()
    if add:
        assert torch.equal(out[m].view(torch.int16), c.out[m].view(torch.int16))
    else:
        assert (out[m].float() == 0).all()


@pytest.mark.parametrize("r", (16, 32, 64))
def test_prefill_gateup(cuda_lib, r):
    c = li.prefill_gateup(r=r)
    rows = np.sort(np.random.default_rng(r).choice(c.T, size=min(c.T, 384), replace=False))
    check(cuda_lib, c, rows)


@pytest.mark.parametrize("N,sgmv", [(8192, False), (8192, True)])
def test_mixed_rank_70b(cuda_lib, N, sgmv):
    c = li.mixed_rank_70b(N=N, sgmv=sgmv)
    rows = np.sort(np.random.default_rng(N).choice(c.T, size=256, replace=False))
    check(cuda_lib, c, rows)


@pytest.mark.parametrize("H,batch,sl", [(1024, 16, 1), (4096, 512, 1), (2049, 16, 8),
                                        (8192, 128, 8), (16384, 16, 1)])
def test_sweep_points(cuda_lib, H, batch, sl):
    c = li.sweep(H=H, batch=batch, seq_len=sl)
    rows = None
    if c.T > 512:
        rows = np.sort(np.random.default_rng(H + batch).choice(c.T, 512, replace=False))
    check(cuda_lib, c, rows)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("T,H,R,L,Ns,add", [
    (1, 64, 16, 1, [64], True),
    (65, 1024, 16, 3, [200], True),
    (130, 2048, 8, 4, [2048], False),
    (64, 4096, 32, 5, [1032, 1024], True),
    (100, 640, 64, 3, [384, 128], False),
    (77, 7, 3, 2, [5], True),          # odd sizes: generic paths
    (300, 512, 24, 2, [256, 104], True),
])
def test_edge_shapes(cuda_lib, dtype, T, H, R, L, Ns, add):
    c = make_case(T, H, R, L, Ns, dtype, seed=T * 13 + H, add=add)
    check(cuda_lib, c)


def test_mixed_ranks_with_zero(cuda_lib):
    c = make_case(400, 1024, 32, 6, [320, 96, 96], torch.bfloat16, seed=19,
                  ranks=[0, 1, 7, 16, 31, 32])
    check(cuda_lib, c)


def test_all_inactive(cuda_lib):
    for add in (True, False):
        c = make_case(100, 256, 16, 2, [256], torch.bfloat16, seed=4, p_neg=1.1, add=add)
        y, out = check(cuda_lib, c)
        assert (y.numpy() == 0).all()
        if add:
            assert torch.equal(out.view(torch.int16), c.out.view(torch.int16))


def test_matches_two_operator_path(cuda_lib):
    """The chained call and the two separate calls agree bit for bit."""
    lg = cuda_lib
    c = li.decode_qkv(512, seed=99)
    y1, o1, _ = gpu_run(lg, c)
    y2, o2, _ = gpu_run_chained(lg, c)
    assert torch.equal(y2, y1)
    assert torch.equal(o2.view(torch.int16), o1.view(torch.int16))


def test_plan_mismatch_writes_nothing(cuda_lib):
    lg = cuda_lib
    c = make_case(50, 128, 16, 3, [64], torch.float16, seed=14)
    plan = lg.new_plan(c.T, c.L)
    lg.lora_group_tokens(c.token_idx.cuda(), c.L, plan)
    y = torch.full((c.T, 16), 7.0, device="cuda")
    out = c.out.cuda()
    A2 = torch.cat([c.A, c.A]).cuda()       # L = 6, the plan has L = 3
    B2 = torch.cat([c.B[0], c.B[0]]).cuda()
    lg.lora_shrink_expand_slice(c.x.cuda(), A2, y, [B2], out, plan, [0])
    torch.cuda.synchronize()
    assert (y.cpu() == 7.0).all()
    assert torch.equal(out.cpu().view(torch.int16), c.out.view(torch.int16))
    _, err = lg.lora_get_error(plan)
    assert err & lg.PLANERR_MISMATCH
