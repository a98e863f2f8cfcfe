"""Input generators and the bench's work formulas (CPU).

The row generator must give the bytes of the whole-tensor generator; the bench's algorithmic
byte and FLOP counts must give the figures the pages and the scope table state: the tiny model
reads 166.9 MB of weights per decode token and costs 5.64 MFLOP of matrix products per prompt
token ("llama.cpp Architecture", Example 13); the 8B shape reads 15.01 GB of BF16 weights and a
512-token prompt costs 7.22 TFLOP."""
import pytest
import torch

import bench
import synthetic as S


@pytest.mark.parametrize("wt", [S.F32, S.F16, S.BF16, S.Q8_0])
def test_weight_rows_equal_the_rows_of_the_whole_tensor(wt):
    shape = (64, 50)
    whole = S.weight_bytes(9, "blk.3.ffn_up.weight", shape, wt)
    rows = [49, 0, 7, 7]
    part = S.weight_rows(9, "blk.3.ffn_up.weight", shape, wt, rows)
    assert torch.equal(whole[rows].view(torch.uint8), part.view(torch.uint8))


def test_bench_work_formulas():
    tiny = S.WORKLOADS["tiny_f32_1seq"]
    assert round(bench.linear_weight_bytes(tiny) / 1e6, 1) == 166.9
    # the pages' per-prompt-token figure counts the layers' matrix products (no output matrix)
    assert round(2 * bench.linear_params_per_layer(tiny.hp) * tiny.hp.n_layer / 1e6, 2) == 5.64
    c3 = S.WORKLOADS["llama8b_bf16_1seq"]
    assert abs(bench.linear_weight_bytes(c3) - 15.0093e9) < 1e6
    fl = bench.prefill_flops(c3.hp, 512, bench.causal_pairs(512), 1)
    assert abs(fl / 1e12 - 7.2167) < 1e-3
    # a decode step at context 640 reads about 15.09 GB
    assert abs(bench.decode_step_bytes(c3, [640], 1) / 1e9 - 15.095) < 0.01
    c5 = S.WORKLOADS["llama8b_bf16_32seq"]
    vis = bench.visible_cells(c5, c5.n_decode)
    assert vis[0] == [2049] * 32
    assert vis[c5.seq_rm_at - 1][0] == 2048 + c5.seq_rm_at
    assert vis[c5.seq_rm_at][0] == (2048 + c5.seq_rm_at) // 2 + 1
