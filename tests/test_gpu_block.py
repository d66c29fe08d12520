"""GPU parity of the whole block (h3_block_forward through the C-ABI)
against the oracle: every row of the tiny block, a seeded 512-row sample of
the full packed-sequence block, determinism and pad invariance."""
import numpy as np
import pytest
import torch

import oracle.h3_oracle as O
from dit_transformer_block_gb300 import inputs as I
from helpers import assert_close_bf16, assert_close_block, np64, sample_rows

pytestmark = pytest.mark.gpu
dev = "cuda"


def gpu_block(h3lib, shape, inp, rope_pairing=0):
    cfg = h3lib.block_config(shape.S, shape.L, shape.D, shape.H, shape.Dh, shape.F,
                             shape.axis_dims, shape.theta, shape.eps_ln, shape.eps_qk,
                             rope_pairing)
    ws = torch.empty(h3lib.block_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    resid = inp["resid"].clone()
    h3lib.block_forward(cfg, inp, resid, inp["mod"], inp["pos"], ws)
    h3lib.check_device_error()
    return resid


def check_block(out_rows, shape, inp, rows=None, what="block", rope_pairing="interleaved"):
    """Compares GPU output rows with the oracle's, with the block tolerance."""
    n = {k: np64(v) if v.is_floating_point() else v.cpu().numpy() for k, v in inp.items()}
    ref, mids = O.block_forward(n["resid"], n["mod"], n["w_qkv"], n["w_o"], n["w_gu"],
                                n["w_down"], n["q_gain"], n["k_gain"], n["pos"], L=shape.L,
                                heads=shape.H, head_dim=shape.Dh, axis_dims=shape.axis_dims,
                                theta=shape.theta, eps_ln=shape.eps_ln, eps_qk=shape.eps_qk,
                                rows=rows, return_intermediates=True, rope_pairing=rope_pairing)
    r_in = n["resid"][:shape.L] if rows is None else n["resid"][rows]
    assert_close_block(np64(out_rows), ref, mids["f"], mids["o"], n["mod"][2], n["mod"][5], r_in,
                       what)


SMALL = [I.TINY,
         I.BlockShape(S=384, L=321, D=768, H=6, Dh=128, F=2048, axis_dims=(32, 48, 48),
                      pos_kind="3d", grid=(2, 10, 16), n_tail=22),
         I.BlockShape(S=64, L=1, D=256, H=2, Dh=128, F=256)]


@pytest.mark.parametrize("shape", SMALL, ids=["tiny", "ragged3d", "one_row"])
def test_block_small(h3lib, shape):
    inp = {k: v.to(dev) for k, v in I.block_inputs(shape, seed=0).items()}
    out = gpu_block(h3lib, shape, inp)
    check_block(out[:shape.L], shape, inp)
    assert torch.equal(out[shape.L:], inp["resid"][shape.L:]), "pad rows written"


@pytest.mark.parametrize("shape", SMALL[:2], ids=["tiny", "ragged3d"])
def test_block_small_split_half_rope(h3lib, shape):
    inp = {k: v.to(dev) for k, v in I.block_inputs(shape, seed=5).items()}
    out = gpu_block(h3lib, shape, inp, rope_pairing=1)
    check_block(out[:shape.L], shape, inp, what="block split-half", rope_pairing="half")
    # the layout matters: the interleaved block gives a different result
    other = gpu_block(h3lib, shape, inp, rope_pairing=0)
    assert not torch.equal(out[:shape.L], other[:shape.L])
    assert torch.equal(out[shape.L:], inp["resid"][shape.L:]), "pad rows written"


def test_block_forward_events_times_every_stage_and_changes_nothing(h3lib):
    # h3_block_forward_events runs the same kernels as h3_block_forward and
    # records one event before every stage and one after the last
    shape = SMALL[1]
    inp = {k: v.to(dev) for k, v in I.block_inputs(shape, seed=4).items()}
    plain = gpu_block(h3lib, shape, inp)
    cfg = h3lib.block_config(shape.S, shape.L, shape.D, shape.H, shape.Dh, shape.F,
                             shape.axis_dims, shape.theta, shape.eps_ln, shape.eps_qk)
    ws = torch.empty(h3lib.block_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    events = [torch.cuda.Event(enable_timing=True) for _ in range(h3lib.BLOCK_STAGES + 1)]
    for e in events:  # create the handles before they are handed to the library
        e.record(stream)
    resid = inp["resid"].clone()
    h3lib.block_forward(cfg, inp, resid, inp["mod"], inp["pos"], ws, events=events)
    h3lib.check_device_error()
    torch.cuda.synchronize()
    assert torch.equal(resid, plain)
    stage = [events[i].elapsed_time(events[i + 1]) for i in range(h3lib.BLOCK_STAGES)]
    total = events[0].elapsed_time(events[-1])
    assert all(t > 0 for t in stage)
    assert abs(sum(stage) - total) <= 1e-3 * total + 1e-3
    # a wrong number of events is refused before anything runs
    with pytest.raises(h3lib.H3Error):
        h3lib.block_forward(cfg, inp, resid, inp["mod"], inp["pos"], ws, events=events[:-1])


def test_block_deterministic_and_pad_invariant(h3lib):
    shape = I.TINY
    inp = {k: v.to(dev) for k, v in I.block_inputs(shape, seed=1).items()}
    a = gpu_block(h3lib, shape, inp)
    b = gpu_block(h3lib, shape, inp)
    assert torch.equal(a, b)
    inp2 = dict(inp)
    r2 = inp["resid"].clone()
    r2[shape.L:] = 1e4
    p2 = inp["pos"].clone()
    p2[shape.L:] = 999
    inp2["resid"], inp2["pos"] = r2, p2
    c = gpu_block(h3lib, shape, inp2)
    assert torch.equal(a[:shape.L], c[:shape.L])


@pytest.mark.parametrize("L", [300, 129])
def test_block_full_width_short_sequence(h3lib, L):
    # the full hidden width (5376, 42 heads, SwiGLU 14336) on a short ragged
    # sequence: every row against the oracle
    S = (L + 63) // 64 * 64
    shape = I.BlockShape(S=S, L=L, D=5376, H=42, Dh=128, F=14336, axis_dims=(32, 48, 48),
                         pos_kind="3d", grid=(31, 24, 79), n_tail=22)
    inp = I.block_inputs(shape, seed=L, device=dev)
    out = gpu_block(h3lib, shape, inp)
    check_block(out[:L], shape, inp, what=f"full-width block L={L}")
    assert torch.equal(out[L:], inp["resid"][L:])


def test_block_valid_rows_unchanged_when_the_buffer_grows(h3lib):
    # the same valid rows in a buffer with 128 more pad rows give the same bits
    shape = I.TINY
    inp = {k: v.to(dev) for k, v in I.block_inputs(shape, seed=2).items()}
    a = gpu_block(h3lib, shape, inp)
    big = I.BlockShape(S=shape.S + 128, L=shape.L, D=shape.D, H=shape.H, Dh=shape.Dh,
                       F=shape.F, axis_dims=shape.axis_dims, theta=shape.theta)
    grow = lambda t, fill: torch.cat([t, torch.full((128,) + tuple(t.shape[1:]), fill,
                                                    dtype=t.dtype, device=dev)])
    inp2 = dict(inp)
    inp2["resid"] = grow(inp["resid"], 3.5)
    inp2["pos"] = grow(inp["pos"], 7)
    b = gpu_block(h3lib, big, inp2)
    assert torch.equal(a[:shape.L], b[:shape.L])
    assert torch.equal(b[shape.L:], inp2["resid"][shape.L:])


@pytest.mark.slow
def test_block_full_size_sampled(h3lib):
    shape = I.FULL
    inp = I.block_inputs(shape, seed=3, device=dev)
    out = gpu_block(h3lib, shape, inp)
    rows = sample_rows(shape.L, 512, 3)
    check_block(out[torch.from_numpy(rows).to(dev)], shape, inp, rows, "block full")
    assert torch.equal(out[shape.L:], inp["resid"][shape.L:])


@pytest.mark.slow
@pytest.mark.parametrize("L", [29034, 87846])
def test_block_stack_length_sweep(h3lib, L):
    """A stack of blocks with independent seeded weights at the short and long
    packed lengths (buffers padded to a multiple of 64): each block is checked
    on sampled rows against the oracle given the GPU's own input to that
    block; the 29,034-row case runs four blocks, the 87,846-row case one."""
    S = (L + 63) // 64 * 64
    shape = I.BlockShape(S=S, L=L, D=5376, H=42, Dh=128, F=14336, axis_dims=(32, 48, 48),
                         pos_kind="3d", grid=(47, 24, 79) if L > 60000 else (16, 24, 79))
    blocks = 4 if L < 60000 else 1
    x = None
    for b in range(blocks):
        inp = I.block_inputs(shape, seed=4 + b + (0 if L < 60000 else 10), device=dev)
        if x is not None:
            inp["resid"] = x
        out = gpu_block(h3lib, shape, inp)
        rows = sample_rows(L, 128, 40 + b)
        check_block(out[torch.from_numpy(rows).to(dev)], shape, inp, rows, f"block {b} L={L}")
        assert torch.equal(out[L:], inp["resid"][L:])
        x = out


def _stack_inputs(shape, nblocks, G=None, seed=20):
    blocks = [{k: v.to(dev) for k, v in I.block_inputs(shape, seed=seed + b).items()}
              for b in range(nblocks)]
    resid = blocks[0]["resid"].clone()
    if G is None:
        mods = torch.stack([b["mod"] for b in blocks]).contiguous()
        seg = None
    else:
        g = torch.Generator(device="cpu")
        g.manual_seed(seed)
        mods = (torch.randn(nblocks, G, 6, shape.D, generator=g) * 0.1).to(dev).contiguous()
        seg = torch.randint(0, G, (shape.S,), generator=g, dtype=torch.int32).to(dev)
    return blocks, resid, mods, seg


def _oracle_stack(shape, blocks, resid, mods, seg):
    W = [tuple(np64(b[k]) for k in ("w_qkv", "w_o", "w_gu", "w_down")) for b in blocks]
    return O.stack_forward(np64(resid), list(np64(mods)), W, [np64(b["q_gain"]) for b in blocks],
                           [np64(b["k_gain"]) for b in blocks], blocks[0]["pos"].cpu().numpy(),
                           L=shape.L, heads=shape.H,
                           head_dim=shape.Dh, axis_dims=shape.axis_dims, theta=shape.theta,
                           seg=None if seg is None else seg.cpu().numpy())


def _cfg(h3lib, shape):
    return h3lib.block_config(shape.S, shape.L, shape.D, shape.H, shape.Dh, shape.F,
                              shape.axis_dims, shape.theta, shape.eps_ln, shape.eps_qk)


@pytest.mark.parametrize("G", [None, 3])
def test_stack_of_four_tiny_blocks(h3lib, G):
    shape = I.TINY
    blocks, resid0, mods, seg = _stack_inputs(shape, 4, G)
    cfg = _cfg(h3lib, shape)
    ws = torch.empty(h3lib.block_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    out = resid0.clone()
    h3lib.stack_forward(cfg, blocks, out, mods, blocks[0]["pos"], ws, seg=seg)
    h3lib.check_device_error()
    ref = _oracle_stack(shape, blocks, resid0, mods, seg)
    assert_close_bf16(np64(out[:shape.L]), ref, "stack")
    r_in = np64(resid0[:shape.L])
    assert_close_bf16(np64(out[:shape.L]) - r_in, ref - r_in, "stack increment")
    assert torch.equal(out[shape.L:], resid0[shape.L:])
    if G is None:
        # the fused block boundary gives the same bits as separate block calls
        seq = resid0.clone()
        for b in range(4):
            h3lib.block_forward(cfg, blocks[b], seq, mods[b], blocks[0]["pos"], ws)
        h3lib.check_device_error()
        assert torch.equal(seq, out)


@pytest.mark.slow
def test_segmented_block_full_size_sampled(h3lib):
    shape = I.FULL
    inp = I.block_inputs(shape, seed=7, device=dev)
    g = torch.Generator(device="cpu")
    g.manual_seed(7)
    mods = (torch.randn(1, 2, 6, shape.D, generator=g) * 0.1).to(dev).contiguous()
    # video tokens in group 0, the trailing audio/text tokens in group 1
    seg = torch.zeros(shape.S, dtype=torch.int32, device=dev)
    seg[shape.L - shape.n_tail:] = 1
    cfg = _cfg(h3lib, shape)
    ws = torch.empty(h3lib.block_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    out = inp["resid"].clone()
    h3lib.stack_forward(cfg, [inp], out, mods, inp["pos"], ws, seg=seg)
    h3lib.check_device_error()
    rows = np.unique(np.concatenate([sample_rows(shape.L, 256, 8),
                                     np.arange(shape.L - shape.n_tail, shape.L)]))
    n = {k: np64(v) if v.is_floating_point() else v.cpu().numpy() for k, v in inp.items()}
    ref, mids = O.block_forward(n["resid"], np64(mods[0]), n["w_qkv"], n["w_o"], n["w_gu"],
                                n["w_down"], n["q_gain"], n["k_gain"], n["pos"], L=shape.L,
                                heads=shape.H, head_dim=shape.Dh, axis_dims=shape.axis_dims,
                                theta=shape.theta, rows=rows, return_intermediates=True,
                                seg=seg.cpu().numpy())
    m = O.modulation_rows(np64(mods[0]), seg.cpu().numpy(), rows)
    from helpers import assert_close_block as acb
    acb(np64(out[torch.from_numpy(rows).to(dev)]), ref, mids["f"], mids["o"], m[:, 2], m[:, 5],
        n["resid"][rows], "segmented block full")
