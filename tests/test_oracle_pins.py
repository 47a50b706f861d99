"""Pins for the CPU oracle: checks against facts that do not come from the
oracle itself (closed forms, library routines, a reformulation, invariants
the pages fix, a hand-worked example and a golden grouping).

Each test is chosen to fail on a plausible slip in the oracle: a transposed
operand or swapped index (one-hot tests), a dropped scale or add term
(hand-worked example, linearity), a wrong adapter or a leaked -1 token
(masked-sum form), an unstable or mis-ordered grouping (library sort,
golden), slice or rank book-keeping (concatenation, zero padding).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import lora_inputs as li

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(t):
    return t.double().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- closed forms

def test_hand_worked_example():
    """T=3, H=2, L=2, R=1; values worked out by hand.

    x = [[1,2],[3,4],[5,6]], A[0] = [[1,-1]], A[1] = [[2,1]], idx = [1,-1,0]
      y[0] = 2*1 + 1*2 = 4,  y[1] = 0 (no LoRA),  y[2] = 1*5 - 1*6 = -1
    B[0] = [[1],[2]], B[1] = [[3],[-1]], out0 = [[10,20],[30,40],[50,60]],
    scale 0.5, add_inputs:
      out[0] = [10 + .5*4*3, 20 + .5*4*(-1)] = [16, 18]
      out[1] = [30, 40]                       (untouched)
      out[2] = [50 + .5*(-1)*1, 60 + .5*(-1)*2] = [49.5, 59]
    """
    x = np.array([[1, 2], [3, 4], [5, 6]], float)
    A = np.array([[[1, -1]], [[2, 1]]], float)
    B = np.array([[[1], [2]], [[3], [-1]]], float)
    out0 = np.array([[10, 20], [30, 40], [50, 60]], float)
    lo, bad = oracle.map_tokens([1, -1, 0], 2)
    assert bad == 0
    y = oracle.shrink(x, A, lo)
    np.testing.assert_array_equal(y, [[4], [0], [-1]])
    out = oracle.expand(y, B, lo, out0, scale=0.5, add=True)
    np.testing.assert_array_equal(out, [[16, 18], [30, 40], [49.5, 59]])
    out_noadd = oracle.expand(y, B, lo, out0, scale=0.5, add=False)
    np.testing.assert_array_equal(out_noadd, [[6, -2], [0, 0], [-0.5, -1]])


def test_shrink_onehot_x_selects_adapter_column():
    """x[t] = e_h  =>  y[t, j] = scale * A[l, j, h]  (catches a transposed A)."""
    g = rng(1)
    L, S, R, H, T = 3, 2, 5, 7, 9
    A = g.standard_normal((L, S * R, H))
    hs = g.integers(0, H, T)
    idx = g.integers(0, L, T)
    x = np.zeros((T, H))
    x[np.arange(T), hs] = 1.0
    y = oracle.shrink(x, A, idx.astype(np.int32), num_slices=S, scale=0.25)
    for t in range(T):
        np.testing.assert_array_equal(y[t], 0.25 * A[idx[t], :, hs[t]])


def test_expand_onehot_y_selects_weight_column():
    """y[t] = e_i  =>  out[t, off+n] = out0 + scale * B[l, n, i]."""
    g = rng(2)
    L, R, T = 3, 6, 8
    Ns, offs, Ntot = [5, 3], [1, 7], 11
    Bs = [g.standard_normal((L, n, R)) for n in Ns]
    i_s = g.integers(0, R, T)
    idx = g.integers(0, L, T).astype(np.int32)
    y = np.zeros((T, 2 * R))
    for t in range(T):
        y[t, i_s[t]] = 1.0       # slice 0 block
        y[t, R + i_s[t]] = 1.0   # slice 1 block
    out0 = g.standard_normal((T, Ntot))
    out = oracle.expand_slice(y, Bs, offs, idx, out0, y_stride=R, scale=2.0, add=True)
    for t in range(T):
        exp = out0[t].copy()
        for s in range(2):
            exp[offs[s]:offs[s] + Ns[s]] += 2.0 * Bs[s][idx[t], :, i_s[t]]
        np.testing.assert_array_equal(out[t], exp)


# ----------------------------------------------------------- library routines

def test_single_adapter_equals_dense_matmul():
    """One adapter, no -1 tokens: shrink = x A^T, expand = out + s * y B^T
    (the torch.mm "single-lora roofline" of vLLM PR #11579)."""
    g = rng(3)
    T, H, R, N = 33, 70, 12, 45
    x = g.standard_normal((T, H))
    A = g.standard_normal((1, R, H))
    B = g.standard_normal((1, N, R))
    out0 = g.standard_normal((T, N))
    lo = np.zeros(T, np.int32)
    y = oracle.shrink(x, A, lo, scale=1.5)
    np.testing.assert_allclose(y, 1.5 * (x @ A[0].T), rtol=1e-12, atol=1e-12)
    out = oracle.expand(y, B, lo, out0, scale=0.75, add=True)
    np.testing.assert_allclose(out, out0 + 0.75 * (y @ B[0].T), rtol=1e-12, atol=1e-12)


def test_masked_sum_formulation():
    """Multi-adapter BGMV equals the masked sum over adapters of dense matmuls
    (the mask formulation of the TPU kernel in vLLM PR #15655)."""
    g = rng(4)
    T, H, R, N, L = 40, 33, 8, 29, 5
    x = g.standard_normal((T, H))
    A = g.standard_normal((L, R, H))
    B = g.standard_normal((L, N, R))
    out0 = g.standard_normal((T, N))
    idx = g.integers(-1, L, T).astype(np.int32)
    lo, _ = oracle.map_tokens(idx, L)
    y = oracle.shrink(x, A, lo, scale=0.5)
    y_ref = sum((idx == l)[:, None] * (x @ A[l].T) for l in range(L)) * 0.5
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)
    out = oracle.expand(y, B, lo, out0, scale=1.25, add=True)
    out_ref = out0 + 1.25 * sum((idx == l)[:, None] * (y @ B[l].T) for l in range(L))
    np.testing.assert_allclose(out, out_ref, rtol=1e-12, atol=1e-12)


def test_group_matches_library_stable_sort():
    g = rng(5)
    for T, L in [(1, 1), (17, 3), (300, 7), (1000, 32)]:
        idx = g.integers(-1, L, T).astype(np.int32)
        gr = oracle.group(idx, L, by_adapter=True, tile=16)
        active = sorted((int(idx[t]), t) for t in range(T) if idx[t] >= 0)
        inactive = [t for t in range(T) if idx[t] < 0]
        assert gr["perm"].tolist() == [t for _, t in active] + inactive
        np.testing.assert_array_equal(gr["count"], np.bincount(idx[idx >= 0], minlength=L))
        np.testing.assert_array_equal(gr["offset"], np.concatenate([[0], np.cumsum(gr["count"])]))
        present = [l for l in range(L) if gr["count"][l] > 0]
        assert gr["group_lora"].tolist() == present
        # tiles cover every position exactly once, in order, never mixing adapters
        covered = []
        for l, p0, n, grp in gr["tiles"].tolist():
            assert 1 <= n <= 16
            ids = {int(idx[gr["perm"][p]]) if idx[gr["perm"][p]] >= 0 else -1
                   for p in range(p0, p0 + n)}
            assert ids == {l}
            covered.extend(range(p0, p0 + n))
        assert covered == list(range(T))


def test_group_golden_aaabcc():
    with open(os.path.join(GOLDEN, "aaabcc_grouping.json")) as f:
        gold = json.load(f)
    for c in gold["cases"]:
        L = c["L"]
        if "idx" in c:
            lo, bad = oracle.map_tokens(c["idx"], L)
            gr = oracle.group(lo, L, by_adapter=True)
        else:
            segs = np.array(c["segments"], np.int32)
            lo, bad, err = oracle.map_segments(segs[:, 0], segs[:, 1], segs[:, 2], c["T"], L)
            assert err == 0
            gr = oracle.group(lo, L, by_adapter=False)
        assert bad == 0
        for k in ("perm", "count", "offset", "group_lora", "group_start", "group_count",
                  "tiles"):
            assert gr[k].tolist() == c[k], (c["name"], k)


# ------------------------------------------------------------------ invariants

def test_bgmv_equals_sgmv_on_same_map():
    """Punica issue #17: BGMV semantics are a strict subset of SGMV's."""
    case = li.prefill_gateup(r=4, H=48, N=40, lens=[5, 1, 9, 3, 4, 2, 7, 6])
    T = case.T
    lo_s, bad, err = oracle.map_segments(case.seg_start, case.seg_len, case.seg_lora, T, case.L)
    assert bad == 0 and err == 0
    lo_b, _ = oracle.map_tokens(case.lora_of_token(), case.L)
    np.testing.assert_array_equal(lo_s, lo_b)
    gs = oracle.group(lo_s, case.L, by_adapter=False)
    gb = oracle.group(lo_b, case.L, by_adapter=True)
    # segments already sorted by adapter: both groupings coincide
    np.testing.assert_array_equal(gs["perm"], gb["perm"])
    np.testing.assert_array_equal(gs["group_count"], gb["group_count"])
    y_s = oracle.shrink(f64(case.x), f64(case.A), lo_s, num_slices=2)
    y_b = oracle.shrink(f64(case.x), f64(case.A), lo_b, num_slices=2)
    np.testing.assert_array_equal(y_s, y_b)


def test_expand_slice_equals_concatenated_expand():
    """vLLM PR #11579 emulates expand_slice by back-to-back expands; with a
    shared y that is one expand into the concatenated weights."""
    g = rng(6)
    T, R, L = 21, 6, 3
    Ns = [8, 5, 11]
    Bs = [g.standard_normal((L, n, R)) for n in Ns]
    y = g.standard_normal((T, R))
    out0 = g.standard_normal((T, sum(Ns)))
    idx = g.integers(-1, L, T).astype(np.int32)
    offs = [0, 8, 13]
    sliced = oracle.expand_slice(y, Bs, offs, idx, out0, y_stride=0, scale=0.5)
    cat = oracle.expand(y, np.concatenate(Bs, axis=1), idx, out0, scale=0.5)
    np.testing.assert_allclose(sliced, cat, rtol=0, atol=0)
    seq = out0.copy()
    for s in range(3):
        seq = oracle.expand_slice(y, [Bs[s]], [offs[s]], idx, seq, y_stride=0, scale=0.5)
    np.testing.assert_array_equal(sliced, seq)


def test_expand_slice_reads_each_slice_y_block():
    """vLLM PR #11579 (num_slices): slice s of a stacked shrink output lives in
    y columns [s*R, (s+1)*R); expand_slice with y_stride = R equals one
    single-slice expand per y column block into that slice's out columns."""
    g = rng(11)
    T, R, L = 17, 5, 3
    Ns = [6, 4, 9]
    offs = [0, 6, 10]
    Bs = [g.standard_normal((L, n, R)) for n in Ns]
    y = g.standard_normal((T, 3 * R + 2))  # ldy > S * R
    out0 = g.standard_normal((T, sum(Ns) + 3))
    idx = g.integers(-1, L, T).astype(np.int32)
    sliced = oracle.expand_slice(y, Bs, offs, idx, out0, y_stride=R, scale=0.7)
    for s in range(3):
        cols = slice(offs[s], offs[s] + Ns[s])
        part = oracle.expand(y[:, s * R:(s + 1) * R].copy(), Bs[s], idx, out0[:, cols].copy(),
                             scale=0.7)
        np.testing.assert_array_equal(sliced[:, cols], part)
    np.testing.assert_array_equal(sliced[:, sum(Ns):], out0[:, sum(Ns):])


def test_expand_slice_leaves_other_columns():
    g = rng(7)
    T, R, L = 9, 4, 2
    B = g.standard_normal((L, 5, R))
    y = g.standard_normal((T, R))
    out0 = g.standard_normal((T, 12))
    idx = g.integers(0, L, T).astype(np.int32)
    out = oracle.expand_slice(y, [B], [3], idx, out0, y_stride=0, add=False)
    np.testing.assert_array_equal(out[:, :3], out0[:, :3])
    np.testing.assert_array_equal(out[:, 8:], out0[:, 8:])


def test_stacked_shrink_equals_separate():
    g = rng(8)
    T, H, R, L, S = 15, 24, 5, 3, 3
    x = g.standard_normal((T, H))
    A = g.standard_normal((L, S * R, H))
    idx = g.integers(-1, L, T).astype(np.int32)
    y = oracle.shrink(x, A, idx, num_slices=S)
    for s in range(S):
        ys = oracle.shrink(x, A[:, s * R:(s + 1) * R, :].copy(), idx)
        np.testing.assert_array_equal(y[:, s * R:(s + 1) * R], ys)


def test_rank_aware_equals_zero_padded():
    """Punica issue #17: padding an adapter's rank up with zeros changes nothing."""
    kw = dict(T=64, H=40, L=6, N=24)
    garbage = li.mixed_rank_70b(pad_fill="garbage", **kw)
    zero = li.mixed_rank_70b(pad_fill="zero", **kw)
    assert torch.equal(garbage.ranks, zero.ranks)
    lo, _ = oracle.map_tokens(garbage.token_idx, garbage.L)
    y_g = oracle.shrink(f64(garbage.x), f64(garbage.A), lo, ranks=garbage.ranks.numpy())
    y_z = oracle.shrink(f64(zero.x), f64(zero.A), lo)
    np.testing.assert_array_equal(y_g, y_z)
    o_g = oracle.expand(y_g, f64(garbage.B[0]), lo, f64(garbage.out), ranks=garbage.ranks.numpy())
    o_z = oracle.expand(y_z, f64(zero.B[0]), lo, f64(zero.out))
    np.testing.assert_array_equal(o_g, o_z)


def test_rank_aware_ignores_padding_in_y_and_b():
    """Punica issue #17 (ranks are not padded to bins): adapter l contributes
    through its first rank(l) coefficients only, whatever y and B hold past
    them.  Brute force with numpy on a tiny case."""
    g = rng(12)
    T, N, R, L = 10, 7, 6, 3
    ranks = np.array([2, 6, 0], np.int32)
    y = g.standard_normal((T, R))
    B = g.standard_normal((L, N, R))
    idx = np.array([0, 1, 2, 1, 0, 2, 2, 0, 1, 0], np.int32)
    out0 = g.standard_normal((T, N))
    got = oracle.expand(y, B, idx, out0, ranks=ranks, scale=1.5)
    for t in range(T):
        l, r = idx[t], ranks[idx[t]]
        ref = out0[t] + 1.5 * (B[l][:, :r] @ y[t, :r])
        np.testing.assert_allclose(got[t], ref, rtol=1e-13, atol=1e-13)


def test_rank_table_clamps():
    """A rank below 0 acts as 0 (no term) and one above R as R (the reading of
    out-of-range ranks: clamped to the stored rows)."""
    g = rng(13)
    T, H, R, N, L = 8, 12, 4, 5, 2
    x = g.standard_normal((T, H))
    A = g.standard_normal((L, R, H))
    B = g.standard_normal((L, N, R))
    idx = np.array([0, 1] * 4, np.int32)
    y = oracle.shrink(x, A, idx, ranks=np.array([-3, 9], np.int32))
    assert (y[idx == 0] == 0).all()
    np.testing.assert_array_equal(y[idx == 1], oracle.shrink(x, A, idx)[idx == 1])
    out0 = g.standard_normal((T, N))
    o = oracle.expand(y, B, idx, out0, ranks=np.array([-3, 9], np.int32))
    np.testing.assert_array_equal(o[idx == 0], out0[idx == 0])
    np.testing.assert_array_equal(o[idx == 1], oracle.expand(y, B, idx, out0)[idx == 1])


def test_inactive_tokens():
    g = rng(9)
    T, H, R, N, L = 12, 10, 4, 6, 2
    x = g.standard_normal((T, H))
    A = g.standard_normal((L, R, H))
    B = g.standard_normal((L, N, R))
    out0 = g.standard_normal((T, N))
    idx = np.array([-1, 0, 1, -1] * 3, np.int32)
    y0 = g.standard_normal((T, R))
    y = oracle.shrink(x, A, idx, y=y0, add=False)
    assert (y[idx < 0] == 0).all()
    y_add = oracle.shrink(x, A, idx, y=y0, add=True)
    np.testing.assert_array_equal(y_add[idx < 0], y0[idx < 0])
    o = oracle.expand(y, B, idx, out0, add=True)
    np.testing.assert_array_equal(o[idx < 0], out0[idx < 0])
    o = oracle.expand(y, B, idx, out0, add=False)
    assert (o[idx < 0] == 0).all()


def test_scale_linearity_and_add_flag():
    g = rng(10)
    T, H, R, N, L = 14, 9, 3, 7, 3
    x = g.standard_normal((T, H))
    A = g.standard_normal((L, R, H))
    B = g.standard_normal((L, N, R))
    idx = g.integers(-1, L, T).astype(np.int32)
    y1 = oracle.shrink(x, A, idx, scale=1.0)
    y3 = oracle.shrink(x, A, idx, scale=3.0)
    np.testing.assert_allclose(y3, 3.0 * y1, rtol=1e-14, atol=1e-14)
    # add=False, then add=True onto zeros, give the same values
    z = np.zeros((T, N))
    a = oracle.expand(y1, B, idx, z, add=False, scale=0.5)
    b = oracle.expand(y1, B, idx, z, add=True, scale=0.5)
    np.testing.assert_array_equal(a, b)
    # shrink add accumulates
    y_acc = oracle.shrink(x, A, idx, y=y1, add=True, scale=1.0)
    np.testing.assert_allclose(y_acc, 2 * y1, rtol=1e-14, atol=1e-14)


# ------------------------------------------------------------------ maps

def test_map_tokens_bad_ids():
    lo, bad = oracle.map_tokens([0, 3, -1, 4, -7, 2], 4)
    assert lo.tolist() == [0, 3, -1, -1, -1, 2]
    assert bad == 2


def test_map_segments_rules():
    # gap, -1 segment, zero-length segment
    lo, bad, err = oracle.map_segments([0, 4, 6, 6], [3, 2, 0, 2], [1, -1, 0, 2], 9, 3)
    assert lo.tolist() == [1, 1, 1, -1, -1, -1, 2, 2, -1] and bad == 0 and err == 0
    # out of range -> ignored, bit 1; overlap -> ignored, bit 2; bad id -> -1
    lo, bad, err = oracle.map_segments([0, 2, 5, 7], [3, 2, 9, 1], [0, 1, 0, 5], 8, 3)
    assert lo.tolist() == [0, 0, 0, -1, -1, -1, -1, -1]
    assert err == 3 and bad == 1


def test_workload_recipes():
    c = li.decode_qkv(T=128)
    assert (c.token_idx == -1).sum().item() == round(0.1 * 128)
    assert c.A.shape == (4, 48, 4096) and [b.shape[1] for b in c.B] == [4096, 1024, 1024]
    assert c.slice_offsets == [0, 4096, 5120] and c.out.shape == (128, 6144)
    p = li.prefill_gateup(r=16)
    assert all(8 <= n <= 2048 for n in p.meta["lens"]) and p.T == sum(p.meta["lens"])
    assert p.seg_lora.tolist() == [0, 0, 0, 1, 2, 2, 3, 3]
    m = li.mixed_rank_70b(T=256, H=64, N=32)
    assert set(m.ranks.tolist()) <= set(li.MIXED_RANKS)
    assert (m.token_idx == -1).sum().item() == round(0.05 * 256)
    s = li.sweep(H=2049, batch=16, seq_len=8)
    assert s.T == 128 and s.seg_len.tolist() == [8] * 16
    assert (s.seg_lora.diff() >= 0).all()
    pp = li.pages_point()
    assert pp.T == 256 and pp.seg_len.tolist() == [16] * 16 and not pp.add
    assert pp.B[0].shape == (4, 2048, 16) and (pp.seg_lora.diff() >= 0).all()
    for name, (Hm, N) in li.MODEL_SHAPES.items():
        c = li.model_shape(name, 100)
        assert c.x.shape == (100, Hm) and c.B[0].shape == (4, N, 16) and c.out.shape == (100, N)
        assert (c.token_idx == -1).sum().item() == 10
