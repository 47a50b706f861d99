"""GPU grouping (BGMV and SGMV plans) against the oracle: bit-exact."""
import json
import os

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def check_plan(lg, plan, T, L, ref, by_adapter, bad_ref=0, err_ref=0):
    v = {k: t.cpu().numpy() for k, t in lg.plan_view(plan, T, L).items()}
    hdr = v["header"]
    assert hdr[lg.HDR["MAGIC"]] == lg.PLAN_MAGIC
    assert hdr[lg.HDR["T"]] == T and hdr[lg.HDR["L"]] == L
    assert hdr[lg.HDR["KIND"]] == (1 if by_adapter else 2)
    assert hdr[lg.HDR["NACTIVE"]] == ref["n_active"]
    G = len(ref["group_lora"])
    assert hdr[lg.HDR["NGROUPS"]] == G
    nt = len(ref["tiles"])
    assert hdr[lg.HDR["NTILES"]] == nt
    assert hdr[lg.HDR["BAD_IDS"]] == bad_ref
    assert hdr[lg.HDR["ERR"]] == err_ref
    np.testing.assert_array_equal(v["perm"], ref["perm"])
    np.testing.assert_array_equal(v["count"], ref["count"])
    np.testing.assert_array_equal(v["offset"], ref["offset"])
    np.testing.assert_array_equal(v["group_lora"][:G], ref["group_lora"])
    np.testing.assert_array_equal(v["group_start"][:G], ref["group_start"])
    np.testing.assert_array_equal(v["group_count"][:G], ref["group_count"])
    np.testing.assert_array_equal(v["tiles"][:nt], ref["tiles"])
    # per-tile row lists: perm[first : first + count], -1 padded
    for k, (l, p0, n, grp) in enumerate(ref["tiles"].tolist()):
        exp = np.full(lg.TILE_TOKENS, -1)
        exp[:n] = ref["perm"][p0:p0 + n]
        np.testing.assert_array_equal(v["tile_rows"][k], exp)
    assert lg.lora_get_error(plan) == (bad_ref, err_ref)


@pytest.mark.parametrize("T,L,lo,seed", [
    (0, 1, -1, 0), (1, 1, 0, 1), (1, 4, -1, 2), (16, 4, -1, 3), (63, 3, -1, 4),
    (64, 2, 0, 5), (65, 7, -1, 6), (1000, 32, -1, 7), (4099, 1024, -1, 8),
    (70001, 5, -1, 9), (2048, 1, 0, 10), (5000, 64, -1, 11)])
def test_group_tokens_matches_oracle(cuda_lib, T, L, lo, seed):
    lg = cuda_lib
    g = np.random.default_rng(seed)
    idx = g.integers(lo, L, T).astype(np.int32)
    plan = lg.new_plan(T, L)
    lg.lora_group_tokens(torch.from_numpy(idx).cuda(), L, plan)
    lof, bad = oracle.map_tokens(idx, L)
    ref = oracle.group(lof, L, by_adapter=True, tile=lg.TILE_TOKENS)
    check_plan(lg, plan, T, L, ref, True, bad)


def test_group_tokens_bad_ids(cuda_lib):
    lg = cuda_lib
    idx = np.array([0, 5, -1, 2, -9, 3, 3, 100, 1] * 40, np.int32)
    L = 4
    plan = lg.new_plan(idx.size, L)
    lg.lora_group_tokens(torch.from_numpy(idx).cuda(), L, plan)
    lof, bad = oracle.map_tokens(idx, L)
    assert bad == 3 * 40
    check_plan(lg, plan, idx.size, L, oracle.group(lof, L, True), True, bad)


def test_group_tokens_zipf_sorted_and_skewed(cuda_lib):
    import lora_inputs as li
    lg = cuda_lib
    for sgmv in (False,):
        c = li.mixed_rank_70b(T=2048, H=16, N=16, sgmv=sgmv)
        plan = lg.new_plan(c.T, c.L)
        lg.lora_group_tokens(c.token_idx.cuda(), c.L, plan)
        lof, bad = oracle.map_tokens(c.token_idx.numpy(), c.L)
        check_plan(lg, plan, c.T, c.L, oracle.group(lof, c.L, True), True, bad)


def segs_case(g, T, S, L, p_gap=0.3, p_neg=0.1, p_zero=0.1):
    starts, lens, loras = [], [], []
    t = 0
    for _ in range(S):
        if g.random() < p_gap:
            t += int(g.integers(1, 5))
        n = 0 if g.random() < p_zero else int(g.integers(1, 40))
        if t + n > T:
            break
        starts.append(t)
        lens.append(n)
        loras.append(-1 if g.random() < p_neg else int(g.integers(0, L)))
        t += n
    return (np.array(starts, np.int32), np.array(lens, np.int32), np.array(loras, np.int32))


@pytest.mark.parametrize("T,S,L,seed", [(0, 0, 1, 0), (10, 0, 2, 1), (50, 3, 2, 2),
                                        (500, 40, 4, 3), (3000, 1500, 8, 4),
                                        (60000, 2500, 16, 5)])
def test_group_segments_matches_oracle(cuda_lib, T, S, L, seed):
    lg = cuda_lib
    g = np.random.default_rng(seed)
    ss, sl, slo = segs_case(g, T, S, L)
    plan = lg.new_plan(T, L)
    lg.lora_group_segments(torch.from_numpy(ss).cuda(), torch.from_numpy(sl).cuda(),
                           torch.from_numpy(slo).cuda(), T, L, plan)
    lof, bad, err = oracle.map_segments(ss, sl, slo, T, L)
    assert err == 0
    check_plan(lg, plan, T, L, oracle.group(lof, L, by_adapter=False), False, bad, err)


def test_group_segments_invalid_entries(cuda_lib):
    lg = cuda_lib
    T, L = 40, 3
    # (2,2) overlaps (0,3); (7,1) and (12,4) start inside (5,9); (-3,2) and
    # (35,100) are out of range; (36,2) is valid but names adapter 7 >= L.
    ss = np.array([0, 2, 5, 7, 12, -3, 30, 29, 35, 36], np.int32)
    sl = np.array([3, 2, 9, 1, 4, 2, 5, 3, 100, 2], np.int32)
    slo = np.array([0, 1, 0, 5, 2, 1, 1, 0, 2, 7], np.int32)
    plan = lg.new_plan(T, L)
    lg.lora_group_segments(torch.from_numpy(ss).cuda(), torch.from_numpy(sl).cuda(),
                           torch.from_numpy(slo).cuda(), T, L, plan)
    lof, bad, err = oracle.map_segments(ss, sl, slo, T, L)
    assert err == 3 and bad == 1
    check_plan(lg, plan, T, L, oracle.group(lof, L, by_adapter=False), False, bad, err)


def test_group_segments_many_chunks_coalesce(cuda_lib):
    """8192 sorted 8-token segments (the sgmv sweep shape) coalesce into <= 4 groups."""
    import lora_inputs as li
    lg = cuda_lib
    c = li.sweep(H=64, batch=8192, seq_len=8)
    plan = lg.new_plan(c.T, c.L)
    lg.lora_group_segments(c.seg_start.cuda(), c.seg_len.cuda(), c.seg_lora.cuda(), c.T, c.L, plan)
    lof, bad, err = oracle.map_segments(c.seg_start.numpy(), c.seg_len.numpy(),
                                        c.seg_lora.numpy(), c.T, c.L)
    ref = oracle.group(lof, c.L, by_adapter=False)
    assert len(ref["group_lora"]) <= 4
    check_plan(lg, plan, c.T, c.L, ref, False, bad, err)


def test_group_golden_aaabcc(cuda_lib):
    lg = cuda_lib
    with open(os.path.join(GOLDEN, "aaabcc_grouping.json")) as f:
        gold = json.load(f)
    for c in gold["cases"]:
        L = c["L"]
        if "idx" in c:
            T = len(c["idx"])
            plan = lg.new_plan(T, L)
            lg.lora_group_tokens(torch.tensor(c["idx"], dtype=torch.int32).cuda(), L, plan)
        else:
            T = c["T"]
            s = torch.tensor(c["segments"], dtype=torch.int32)
            plan = lg.new_plan(T, L)
            lg.lora_group_segments(s[:, 0].contiguous().cuda(), s[:, 1].contiguous().cuda(),
                                   s[:, 2].contiguous().cuda(), T, L, plan)
        v = {k: t.cpu().numpy() for k, t in lg.plan_view(plan, T, L).items()}
        G = len(c["group_lora"])
        assert v["perm"].tolist() == c["perm"], c["name"]
        assert v["count"].tolist() == c["count"]
        assert v["offset"].tolist() == c["offset"]
        assert v["group_lora"][:G].tolist() == c["group_lora"]
        assert v["group_start"][:G].tolist() == c["group_start"]
        assert v["group_count"][:G].tolist() == c["group_count"]
        nt = len(c["tiles"])
        assert v["header"][lg.HDR["NTILES"]] == nt
        assert v["tiles"][:nt].tolist() == c["tiles"]
        for k, (l, p0, n, grp) in enumerate(c["tiles"]):
            assert v["tile_rows"][k].tolist() == c["perm"][p0:p0 + n] + [-1] * (lg.TILE_TOKENS - n)
