"""The one-launch decode pair (lora_bgmv_fused_shrink_expand_slice) against the
oracle, element by element, with the bounds of helpers.py: y within the
fp32-accumulation bound, out within one ulp of the oracle's expand of the
GPU's own y, and out end to end within the output type's tolerance."""
import numpy as np
import pytest
import torch

import lora_inputs as li
from helpers import assert_close, assert_expand_ulp, assert_y_fp32, f64, oracle_run
from test_gpu_bgmv import bgmv_run, inactive_rows_ok
from test_gpu_ops import make_case, skewed_idx

pytestmark = pytest.mark.gpu


def fused_run(lg, case, dev="cuda", y_fill=float("nan")):
    """The one-launch path on the GPU.  Returns (y, out) on the host."""
    out = case.out.to(dev)
    idx = case.token_idx.to(dev) if case.token_idx is not None else None
    ranks = case.ranks.to(dev) if case.ranks is not None else None
    y = torch.full((case.T, case.num_slices * case.R), y_fill, dtype=torch.float32, device=dev)
    lg.lora_bgmv_fused_shrink_expand_slice(
        case.x.to(dev), case.A.to(dev), y, [b.to(dev) for b in case.B], out, case.slice_offsets,
        idx, ranks=ranks, scale_shrink=case.shrink_scale, scale_expand=case.scale,
        add_inputs=case.add)
    torch.cuda.synchronize()
    return y.cpu(), out.cpu()


def check(lg, case):
    y, out = fused_run(lg, case)
    _, o_ref = oracle_run(case)
    assert_y_fp32(y, case, None, f"{case.name} fused")
    assert_expand_ulp(out, y, case, None, f"{case.name} fused")
    assert_close(out, o_ref, case.dtype, f"{case.name} fused out")
    inactive_rows_ok(case, y, out)
    return y, out


@pytest.mark.parametrize("T", [t for t in li.DECODE_T if t <= 256] + [1, 97, 255])
@pytest.mark.parametrize("add", [True, False])
def test_decode_qkv(cuda_lib, T, add):
    c = li.decode_qkv(T) if T in li.DECODE_T else li.decode_qkv(T, seed=T)
    c.add = add
    check(cuda_lib, c)


def test_bgmv_small(cuda_lib):
    check(cuda_lib, li.bgmv_small())


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("T,H,R,L,Ns,ranks", [
    (1, 64, 16, 1, [64], None),              # one token, one K stage
    (129, 520, 8, 3, [200], None),           # ragged tile, H not a multiple of 64, rank 8
    (256, 128, 32, 2, [64, 64], None),       # H of two stages, rank 32
    (200, 2048, 16, 5, [256, 104], [16, 0, 7, 16, 1]),  # rank 0 and odd ranks
    (65, 8192, 8, 8, [136], None),           # 8 adapters, long K, ragged 8-column tail
    (256, 4096, 32, 4, [4096, 1024, 1024], [32, 24, 8, 32]),  # q/k/v at rank 32 (W = 96)
    (100, 1000, 24, 2, [512, 512, 512, 512], None),  # four slices, W = 96, H % 64 != 0
    (100, 1024, 16, 8, [256, 128, 128], None),  # 24 (adapter, slice) units: more than the clusters
    (40, 16384, 8, 2, [64], None),           # four passes of K stages per CTA
])
@pytest.mark.parametrize("add", [False, True])
def test_edge_shapes(cuda_lib, dtype, T, H, R, L, Ns, ranks, add):
    c = make_case(T, H, R, L, Ns, dtype, seed=T * 5 + H + R, add=add, ranks=ranks)
    check(cuda_lib, c)


@pytest.mark.parametrize("T,L,counts", [(256, 4, [0, 0, 256, 0]), (256, 4, [250, 1, 0, 5]),
                                        (100, 8, [0, 10, 10, 10, 10, 10, 10, 10]),
                                        (200, 8, [0, 0, 0, 0, 0, 0, 0, 180]),
                                        (130, 3, [0, 130, 0])])
def test_skewed_and_absent_adapters(cuda_lib, T, L, counts):
    """All tokens on one adapter (four 64-token shrink groups), adapters with
    no token at all (with 8 adapters and 3 slices a cluster's first unit has
    none and its second some)."""
    c = make_case(T, 1024, 16, L, [384, 128, 128] if L == 8 else [384, 128], torch.bfloat16,
                  seed=T + L)
    c.token_idx = skewed_idx(T, counts, seed=T)
    check(cuda_lib, c)


def test_bad_ids_and_all_inactive(cuda_lib):
    c = make_case(200, 512, 16, 3, [256], torch.float16, seed=5)
    c.token_idx[::7] = 3
    c.token_idx[::11] = -5
    check(cuda_lib, c)
    for add in (False, True):
        c = make_case(150, 256, 16, 2, [256], torch.bfloat16, seed=4, p_neg=1.1, add=add)
        check(cuda_lib, c)


def test_single_adapter_no_index(cuda_lib):
    """token_idx = NULL: every token uses adapter 0."""
    for T, H, R, N, add in [(256, 2048, 16, 2048, False), (77, 1536, 16, 2048, True)]:
        c = make_case(T, H, R, 1, [N], torch.float16, seed=T + R, add=add, p_neg=0.0)
        c.token_idx = None
        y, out = check(cuda_lib, c)
        o_ref = (f64(c.out) if add else 0) + c.scale * (f64(y) @ f64(c.B[0][0]).T)
        assert_close(out, o_ref, c.dtype, "dense out")


def test_equals_two_launch_form(cuda_lib):
    """Same y (up to the order of the fp32 additions) and out as the chained pair."""
    lg = cuda_lib
    c = li.decode_qkv(256, seed=77)
    y_f, o_f = fused_run(lg, c)
    y_p, o_p = bgmv_run(lg, c)
    mag = np.abs(f64(y_p)) + 1.0
    assert (np.abs(f64(y_f) - f64(y_p)) <= 2e-5 * mag).all()
    assert_close(o_f, f64(o_p), c.dtype, "out fused vs pair")


def test_repeated_and_graph_replayed(cuda_lib):
    """Two calls in a row, then the call captured in a CUDA graph and replayed
    (a cooperative kernel node): every result within the oracle's bounds."""
    lg = cuda_lib
    c = li.decode_qkv(128, seed=3)
    c.add = False
    y1, o1 = fused_run(lg, c)
    y2, o2 = fused_run(lg, c)
    assert_y_fp32(y1, c, None, "repeat")
    assert_expand_ulp(o1, y1, c, None, "repeat")
    # y's partials are added in a fixed order: the same bits every run
    assert torch.equal(y1, y2) and torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    dev = "cuda"
    x, A = c.x.to(dev), c.A.to(dev)
    Bs = [b.to(dev) for b in c.B]
    idx = c.token_idx.to(dev)
    out = c.out.to(dev)
    y = torch.full((c.T, 48), float("nan"), device=dev)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        lg.lora_bgmv_fused_shrink_expand_slice(x, A, y, Bs, out, c.slice_offsets, idx,
                                               scale_shrink=c.shrink_scale, scale_expand=c.scale,
                                               add_inputs=False)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        lg.lora_bgmv_fused_shrink_expand_slice(x, A, y, Bs, out, c.slice_offsets, idx,
                                               scale_shrink=c.shrink_scale, scale_expand=c.scale,
                                               add_inputs=False)
    y.fill_(float("nan"))
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert_y_fp32(y.cpu(), c, None, "graph")
    assert_expand_ulp(out.cpu(), y.cpu(), c, None, "graph")
    _, o_ref = oracle_run(c)
    assert_close(out.cpu(), o_ref, c.dtype, "graph out")


def test_unsupported_shapes(cuda_lib):
    lg = cuda_lib
    for T, R in [(257, 16), (64, 48)]:
        c = make_case(T, 256, R, 2, [128], torch.float16, seed=T + R)
        with pytest.raises(lg.LoraError) as e:
            fused_run(lg, c)
        assert e.value.status == 2
    # an empty batch is a no-op
    c = make_case(1, 256, 16, 2, [128], torch.float16, seed=1)
    dev = "cuda"
    lg.lora_bgmv_fused_shrink_expand_slice(
        torch.empty(0, 256, dtype=torch.float16, device=dev), c.A.to(dev),
        torch.empty(0, 16, device=dev), [c.B[0].to(dev)],
        torch.empty(0, 128, dtype=torch.float16, device=dev), [0],
        torch.empty(0, dtype=torch.int32, device=dev))
