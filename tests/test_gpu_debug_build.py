"""The LORA_DEBUG build (liblora_gemv_debug.so): the same kernels with
device-side bounds checks on every plan entry an operator reads.

- On valid plans it gives bit-for-bit the results of the default build and
  raises no error bit.
- On a plan whose token rows and adapter ids were corrupted by hand, it sets
  LORA_PLANERR_BOUNDS in the plan's error word, where the default build
  stays silent.  Both builds skip the bad entries: the operands are views of
  buffers with spare rows past T, and a corrupted row that points just past
  T would land there, so the spare rows must come back unchanged.
Nothing here faults: the corrupted rows stay inside the padded buffers, and
every build already treats rows outside [0, T) as absent."""
import pytest
import torch

import lora_gemv_gb300 as lg
import lora_inputs as li
from lora_gemv_gb300 import build as lgbuild
from test_gpu_ops import make_case

pytestmark = pytest.mark.gpu

PAD = 8  # spare rows past T in every operand buffer


@pytest.fixture(scope="module")
def debug_path(cuda_lib):
    path = lgbuild.build(debug=True)
    yield path
    lg.use_library(None)


def padded(t, dev="cuda", fill=0.0):
    buf = torch.full((t.shape[0] + PAD,) + tuple(t.shape[1:]), fill, dtype=t.dtype, device=dev)
    buf[:t.shape[0]] = t.to(dev)
    return buf


def run(case, library, corrupt=False):
    """Grouping, shrink and expand_slice through `library`.  Returns the
    y and out buffers (with their spare rows) and the plan's error words."""
    lg.use_library(library)
    dev = "cuda"
    T, L = case.T, case.L
    xb = padded(case.x)
    yb = torch.full((T + PAD, case.num_slices * case.R), 7.0, device=dev)
    ob = padded(case.out, fill=3.0)
    Bs = [b.to(dev) for b in case.B]
    idx = case.token_idx.to(dev)
    ranks = case.ranks.to(dev) if case.ranks is not None else None
    plan = lg.new_plan(T, L, dev)
    lg.lora_group_tokens(idx, L, plan)
    if corrupt:
        lay = lg.lora_plan_layout(T, L)
        rows = plan[lay["tile_rows"]:lay["tile_rows"] + 4 * 64 * 2].view(torch.int32)
        rows[0] = T        # just past the last token: lands in the spare rows if used
        rows[1] = -7       # below -1
        rows[64 + 3] = T + 2
        tiles = plan[lay["tiles"]:lay["tiles"] + 16 * 2].view(torch.int32)
        tiles[4] = L + 1   # the second tile's adapter id
    lg.lora_shrink(xb[:T], case.A.to(dev), yb[:T], plan, num_slices=case.num_slices, ranks=ranks,
                   scale=case.shrink_scale)
    lg.lora_expand_slice(yb[:T], Bs, ob[:T], plan, case.slice_offsets, y_slice_stride=case.R,
                         ranks=ranks, scale=case.scale, add_inputs=case.add)
    bad, err = lg.lora_get_error(plan)
    torch.cuda.synchronize()
    out = (yb.cpu(), ob.cpu(), bad, err)
    lg.use_library(None)
    return out


def cases():
    c1 = li.decode_qkv(128, seed=41)                                  # warp expand, r = 16
    c2 = make_case(200, 1024, 64, 3, [512, 256], torch.bfloat16, seed=42, add=False)  # tc expand
    c3 = make_case(96, 512, 32, 2, [256], torch.float16, seed=43, ranks=[32, 5])
    return [c1, c2, c3]


@pytest.mark.parametrize("k", range(3))
def test_debug_build_matches_default_on_valid_plans(debug_path, k):
    c = cases()[k]
    y_d, o_d, bad_d, err_d = run(c, debug_path)
    y_r, o_r, bad_r, err_r = run(c, None)
    assert err_d == 0 and err_r == 0
    assert bad_d == bad_r
    assert torch.equal(y_d, y_r)
    assert torch.equal(o_d.view(torch.int16), o_r.view(torch.int16))


@pytest.mark.parametrize("k", range(3))
def test_corrupted_plan_is_counted_and_skipped(debug_path, k):
    c = cases()[k]
    T = c.T
    y_d, o_d, _, err_d = run(c, debug_path, corrupt=True)
    y_r, o_r, _, err_r = run(c, None, corrupt=True)
    assert err_d & lg.PLANERR_BOUNDS
    assert not err_r & lg.PLANERR_BOUNDS
    for y, o in ((y_d, o_d), (y_r, o_r)):
        assert (y[T:] == 7.0).all()      # spare rows untouched
        assert (o[T:].float() == 3.0).all()
    # both builds skip the same entries: identical results
    assert torch.equal(y_d, y_r)
    assert torch.equal(o_d.view(torch.int16), o_r.view(torch.int16))
