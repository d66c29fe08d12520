"""The seeded input recipe (CPU): the packed-sequence positions, the pad rows
and the reproducibility the parity tests rely on."""
import torch

from dit_transformer_block_gb300 import inputs as I


def test_positions_3d_walk_the_grid_then_the_tail():
    S, L, grid, n_tail = 64, 50, (2, 3, 5), 20
    pos = I.positions_3d(S, L, grid=grid, n_tail=n_tail)
    T, Hh, W = grid
    for i in range(L - n_tail):  # video tokens: (t, h, w) row-major cells
        assert pos[i].tolist() == [i // (Hh * W), (i // W) % Hh, i % W]
    for i in range(n_tail):  # trailing tokens continue after the last t
        assert pos[L - n_tail + i].tolist() == [T + i] * 3
    assert bool((pos[L:] == 0).all())


def test_full_workload_positions():
    # 58,736 video tokens fill 30 whole t-slices of 24 x 79 and 1,856 cells of
    # slice 30; the 22 audio/text tokens take t = h = w = 31 .. 52
    pos = I.positions_3d(I.FULL.S, I.FULL.L)
    v = I.FULL.L - 22
    assert v == 58736 and v == 30 * 24 * 79 + 1856
    assert pos[v - 1].tolist() == [30, 1855 // 79, 1855 % 79]
    assert pos[v].tolist() == [31, 31, 31] and pos[I.FULL.L - 1].tolist() == [52, 52, 52]


def test_positions_1d():
    pos = I.positions_1d(10, 7)
    assert pos[:7, 0].tolist() == list(range(7))
    assert bool((pos[:, 1:] == 0).all()) and bool((pos[7:] == 0).all())


def test_block_inputs_are_seeded_and_pad_rows_are_garbage():
    a = I.block_inputs(I.TINY, seed=11)
    b = I.block_inputs(I.TINY, seed=11)
    c = I.block_inputs(I.TINY, seed=12)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    assert not torch.equal(a["w_qkv"], c["w_qkv"])
    # the valid residual rows are bf16 values handed over as FP32
    r = a["resid"][:I.TINY.L]
    assert torch.equal(r, r.to(torch.bfloat16).float())
    # the pad rows hold fresh garbage (drawn last, after every other tensor)
    assert a["resid"][I.TINY.L:].abs().sum() > 0
    assert a["mod"].dtype == torch.float32 and a["w_o"].dtype == torch.bfloat16
