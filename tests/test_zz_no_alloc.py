"""lora_shrink_expand_slice_noalloc against the ordinary entry points.

The no-allocation entry point serves callers that are handed their input and
output buffers and cannot allocate the plan buffer themselves (a plugin whose
host owns all device memory, or a serving loop that must not call cudaMalloc
because it can synchronise the device).  It keeps the token grouping in a
fixed device array owned by the library.  Its results must be those of
lora_group_tokens followed by lora_shrink_expand_slice on a caller-allocated
plan, call after call: the array keeps the previous call's plan, so two calls
in a row with different batches check that nothing of the first one leaks
into the second.

This file is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

import lora_inputs as li
from helpers import assert_close

pytestmark = pytest.mark.gpu


def planned(lg, c, dev):
    """The ordinary path: a caller-allocated plan, then the chained pair."""
    plan = lg.new_plan(c.T, c.L, dev)
    lg.lora_group_tokens(c.token_idx.to(dev), c.L, plan)
    y = torch.full((c.T, c.num_slices * c.R), float("nan"), device=dev)
    out = c.out.to(dev)
    lg.lora_shrink_expand_slice(c.x.to(dev), c.A.to(dev), y, [b.to(dev) for b in c.B], out, plan,
                                c.slice_offsets, scale_shrink=c.shrink_scale,
                                scale_expand=c.scale, add_inputs=c.add)
    torch.cuda.synchronize()
    return y.cpu(), out.cpu()


def noalloc(lg, c, dev):
    y = torch.full((c.T, c.num_slices * c.R), float("nan"), device=dev)
    out = c.out.to(dev)
    lg.lora_shrink_expand_slice_noalloc(c.token_idx.to(dev), c.x.to(dev), c.A.to(dev), y,
                                        [b.to(dev) for b in c.B], out, c.slice_offsets,
                                        scale_shrink=c.shrink_scale, scale_expand=c.scale,
                                        add_inputs=c.add)
    torch.cuda.synchronize()
    return y.cpu(), out.cpu()


def test_noalloc_matches_planned_path_two_calls_in_a_row(cuda_lib):
    lg = cuda_lib
    dev = "cuda"
    # a large decode batch, then a smaller one with other adapters idle: the
    # second call must not see any of the first call's plan
    first = li.decode_qkv(1024, seed=4242)
    second = li.decode_qkv(200, seed=4243, L=6)
    act = second.token_idx >= 0
    second.token_idx[act] = 2 + second.token_idx[act] % 4   # adapters 2..5 only
    for c in (first, second):
        y_ref, o_ref = planned(lg, c, dev)
        y, o = noalloc(lg, c, dev)
        assert_close(y, y_ref.double().numpy(), c.dtype, f"{c.name} noalloc y")
        assert_close(o, o_ref.double().numpy(), c.dtype, f"{c.name} noalloc out")
        # the same kernels on the same grouping: identical bits
        assert torch.equal(y, y_ref)
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        inactive = (c.token_idx == -1).numpy()
        assert (y.numpy()[inactive] == 0).all()
        assert torch.equal(o[inactive].view(torch.int16), c.out[inactive].view(torch.int16))


def test_noalloc_rejects_batches_above_its_limit(cuda_lib):
    lg = cuda_lib
    T = lg.NOALLOC_MAX_TOKENS + 1
    c = li.decode_qkv(16)
    x = torch.zeros(T, c.H, dtype=c.dtype, device="cuda")
    idx = torch.zeros(T, dtype=torch.int32, device="cuda")
    y = torch.zeros(T, c.num_slices * c.R, device="cuda")
    out = torch.zeros(T, c.N_total, dtype=c.dtype, device="cuda")
    with pytest.raises(lg.LoraError) as e:
        lg.lora_shrink_expand_slice_noalloc(idx, x, c.A.cuda(), y, [b.cuda() for b in c.B], out,
                                            c.slice_offsets)
    assert e.value.status == 2 and "LORA_NOALLOC_MAX_TOKENS" in str(e.value)
    assert np.all(out.cpu().float().numpy() == 0)
