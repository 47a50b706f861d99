"""The benchmark's algorithmic work formulas (the numerators of every
roofline fraction), checked on a hand-worked batch."""
import torch


def test_decode_algorithmic_work_hand_example():
    import bench
    # 4 tokens: adapters 0, -1, 1, 0 -> 3 active tokens, 2 adapters used.
    # q/k/v workload: H = 4096, S = 3 slices of rank 16, N_tot = 6144, 2-byte elements.
    idx = torch.tensor([0, -1, 1, 0], dtype=torch.int32)
    sh_bytes, sh_flops, ex_bytes, ex_flops = bench.algorithmic(idx)
    # shrink: x rows of active tokens + live A rows of used adapters + y written (fp32)
    assert sh_bytes == 3 * 4096 * 2 + 2 * 48 * 4096 * 2 + 4 * 48 * 4
    assert sh_flops == 2 * 4096 * 48 * 3
    # expand_slice: y rows read + live B rows of used adapters + out read and written
    assert ex_bytes == 3 * 48 * 4 + 2 * 6144 * 16 * 2 + 2 * 3 * 6144 * 2
    assert ex_flops == 2 * 6144 * 16 * 3


def test_decode_algorithmic_work_all_inactive():
    import bench
    idx = torch.full((8,), -1, dtype=torch.int32)
    sh_bytes, sh_flops, ex_bytes, ex_flops = bench.algorithmic(idx)
    assert sh_flops == 0 and ex_flops == 0 and ex_bytes == 0
    assert sh_bytes == 8 * 48 * 4  # y rows are still written (zeros)


def test_chained_work_counts_y_once():
    import bench
    idx = torch.tensor([0, -1, 1, 0], dtype=torch.int32)
    sh_bytes, sh_flops, ex_bytes, ex_flops = bench.algorithmic(idx)
    fu_bytes, fu_flops = bench.algorithmic_fused(idx)
    # the expand's y re-read (3 active tokens x 48 fp32) is not counted again
    assert fu_bytes == sh_bytes + ex_bytes - 3 * 48 * 4
    assert fu_flops == sh_flops + ex_flops


def test_segment_work_hand_example():
    import bench
    # T = 10 tokens, H = 8, N = 6 per slice, r = 2, S = 2 slices, U = 3 adapters
    sh_b, sh_f, ex_b, ex_f = bench.segment_work(10, 8, 6, 2, 2, 3)
    assert sh_b == 10 * 8 * 2 + 3 * 2 * 2 * 8 * 2 + 10 * 2 * 2 * 4
    assert sh_f == 2 * 10 * 8 * 2 * 2
    assert ex_b == 10 * 2 * 2 * 4 + 3 * 2 * 6 * 2 * 2 + 2 * 10 * 2 * 6 * 2
    assert ex_f == 2 * 10 * 2 * 6 * 2


def test_single_slice_work_hand_example():
    import bench
    # 7 of 9 tokens active, 2 adapters used, H = 16, N = 5, r = 4
    sh_b, ex_add = bench.single_slice_work(7, 9, 2, 16, 5, 4, add=True)
    assert sh_b == 7 * 16 * 2 + 2 * 4 * 16 * 2 + 9 * 4 * 4
    assert ex_add == 7 * 4 * 4 + 2 * 5 * 4 * 2 + 2 * 7 * 5 * 2
    _, ex_noadd = bench.single_slice_work(7, 9, 2, 16, 5, 4, add=False)
    assert ex_noadd == 7 * 4 * 4 + 2 * 5 * 4 * 2 + 9 * 5 * 2
