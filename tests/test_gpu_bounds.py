"""Out-of-bounds write checks through the C-ABI: every output (and in-place
operand) is a view into a larger buffer whose 256-byte margins before and
after hold a sentinel; after each call the margins must be untouched and, where
the entry point promises it, so must the pad rows >= L. Shapes are ragged
(L < S, L not a multiple of 128) so the kernels' tail handling is exercised."""
import pytest
import torch

from dit_transformer_block_gb300 import inputs as I

pytestmark = pytest.mark.gpu
dev = "cuda"
MARGIN = 256  # bytes on each side


class Guarded:
    """A tensor of `shape` inside a buffer with sentinel margins."""

    def __init__(self, shape, dtype, fill=None):
        es = torch.empty(0, dtype=dtype).element_size()
        self.g = MARGIN // es
        n = 1
        for d in shape:
            n *= d
        self.n = n
        self.buf = torch.empty(self.g * 2 + n, dtype=dtype, device=dev)
        if dtype == torch.uint8:
            self.buf.fill_(0xA5)
        elif dtype == torch.int32:
            self.buf.fill_(-123456)
        else:
            self.buf.fill_(-7.25)
        self.t = self.buf[self.g:self.g + n].view(*shape)
        if fill is not None:
            self.t.copy_(fill)
        self.head = self.buf[:self.g].clone()
        self.tail = self.buf[self.g + n:].clone()

    def check(self, what):
        assert torch.equal(self.buf[:self.g], self.head), f"{what}: write before the tensor"
        assert torch.equal(self.buf[self.g + self.n:], self.tail), f"{what}: write past the tensor"


def rnd(*shape, std=1.0, seed=0):
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    return (torch.randn(*shape, generator=g, device=dev) * std)


def test_projection_outputs_stay_in_bounds(h3lib):
    S, L, K = 300, 257, 192
    x = rnd(S, K).to(torch.bfloat16)
    w = rnd(512, K, std=0.02, seed=1).to(torch.bfloat16)
    y = Guarded((S, 512), torch.bfloat16)
    h3lib.linear(x, w, y.t, L)
    wgu = rnd(2 * 256, K, std=0.02, seed=2).to(torch.bfloat16)
    u = Guarded((S, 256), torch.bfloat16)
    h3lib.linear_swiglu(x, wgu, u.t, L)
    r = Guarded((S, 512), torch.float32, fill=rnd(S, 512, seed=3))
    r_pad = r.t[L:].clone()
    h3lib.linear_residual(x, w, r.t, rnd(512, seed=4), L)
    H = 2
    wqkv = rnd(3 * H * 128, K, std=0.02, seed=5).to(torch.bfloat16)
    pos = I.positions_3d(S, L, grid=(3, 5, 12), n_tail=L - 180).to(dev)
    tab = Guarded((S, 64, 2), torch.float32)
    h3lib.rope_table(pos, (32, 48, 48), tab.t, L)
    ones = torch.ones(128, device=dev)
    for pairing in (0, 1):
        qkv = Guarded((S, 3 * H * 128), torch.bfloat16)
        h3lib.linear_qk_norm_rope(x, wqkv, qkv.t, ones, ones, tab.t, (32, 48, 48), L,
                                  pairing=pairing)
        h3lib.check_device_error()
        qkv.check(f"linear_qk_norm_rope pairing {pairing}")
        assert bool((qkv.t[L:] == -7.25).all())
    h3lib.check_device_error()
    for g, what in ((y, "linear"), (u, "linear_swiglu"), (r, "linear_residual"),
                    (tab, "rope_table")):
        g.check(what)
    assert bool((y.t[L:] == -7.25).all()) and bool((u.t[L:] == -7.25).all())
    assert torch.equal(r.t[L:], r_pad)
    assert bool((tab.t[L:] == -7.25).all())


def test_attention_outputs_stay_in_bounds(h3lib):
    S, L, H = 300, 259, 3
    q, k, v = (rnd(S, H, 128, seed=s).to(torch.bfloat16) for s in (6, 7, 8))
    nq = (L + 127) // 128
    o = Guarded((S, H, 128), torch.bfloat16)
    h3lib.attention_varlen(q, k, v, o.t, L)
    h3lib.check_device_error()
    o.check("attention")
    assert bool((o.t[L:] == -7.25).all())
    for skip in (0.0, 1e-3):
        o = Guarded((S, H, 128), torch.bfloat16)
        kept = Guarded((nq, H), torch.int32)
        h3lib.attention_varlen_skip(q, k, v, o.t, L, skip_eps=skip, kept=kept.t)
        h3lib.check_device_error()
        o.check(f"attention skip_eps={skip}")
        kept.check(f"kept tiles skip_eps={skip}")
        assert bool((o.t[L:] == -7.25).all())
    ops = h3lib.sage_quantize(q, k, v, L)
    o = Guarded((S, H, 128), torch.bfloat16)
    h3lib.attention_fp8(ops, o.t, L)
    h3lib.check_device_error()
    o.check("attention_fp8")
    assert bool((o.t[L:] == -7.25).all())
    for skip in (0.0, 1e-3):
        o = Guarded((S, H, 128), torch.bfloat16)
        kept = Guarded((nq, H), torch.int32)
        h3lib.attention_fp8_skip(ops, o.t, L, skip_eps=skip, kept=kept.t)
        h3lib.check_device_error()
        o.check(f"attention_fp8 skip_eps={skip}")
        kept.check(f"fp8 kept tiles skip_eps={skip}")
        assert bool((o.t[L:] == -7.25).all())


def test_elementwise_outputs_stay_in_bounds(h3lib):
    S, L, H, D = 200, 131, 3, 640
    pos = I.positions_3d(S, L, grid=(3, 5, 12), n_tail=0).to(dev)
    ones = torch.ones(128, device=dev)
    for pairing in (0, 1):
        q = Guarded((S, H, 128), torch.bfloat16, fill=rnd(S, H, 128, seed=9))
        k = Guarded((S, H, 128), torch.bfloat16, fill=rnd(S, H, 128, seed=10))
        q_pad, k_pad = q.t[L:].clone(), k.t[L:].clone()
        h3lib.qk_norm_rope(q.t, k.t, ones, ones, pos, (32, 48, 48), L, pairing=pairing)
        h3lib.check_device_error()
        q.check("qk_norm_rope q")
        k.check("qk_norm_rope k")
        assert torch.equal(q.t[L:], q_pad) and torch.equal(k.t[L:], k_pad)
    r = Guarded((S, D), torch.float32, fill=rnd(S, D, seed=11))
    r_pad = r.t[L:].clone()
    h = Guarded((S, D), torch.bfloat16)
    mod = rnd(6, D, std=0.1, seed=12)
    h3lib.mod_norm_residual(r.t, rnd(S, D, seed=13).to(torch.bfloat16), mod[2], mod[3], mod[4],
                            h.t, L)
    gu = rnd(S, 2 * 256, seed=14).to(torch.bfloat16)
    u = Guarded((S, 256), torch.bfloat16)
    h3lib.swiglu(gu, u.t, L)
    xq = rnd(S, D, seed=15).to(torch.bfloat16)
    codes = Guarded((S, D), torch.uint8)
    scales = Guarded((S,), torch.float32)
    h3lib.quantize_fp8_rows(xq, codes.t, scales.t)
    frames = rnd(1, 3, 2, 6, 10, seed=16).clamp(-1.2, 1.2)
    out8 = Guarded((1, 2, 6, 10, 3), torch.uint8)
    h3lib.frames_to_u8(frames, out8.t)
    h3lib.check_device_error()
    for g, what in ((r, "mod_norm_residual resid"), (h, "mod_norm_residual normed"),
                    (u, "swiglu"), (codes, "quantize_fp8_rows codes"),
                    (scales, "quantize_fp8_rows scales"), (out8, "frames_to_u8")):
        g.check(what)
    assert torch.equal(r.t[L:], r_pad)
    assert bool((h.t[L:] == -7.25).all()) and bool((u.t[L:] == -7.25).all())


@pytest.mark.parametrize("fp8", [False, True])
def test_block_writes_only_resid_rows_and_workspace(h3lib, fp8):
    shape = I.BlockShape(S=384, L=321, D=768, H=6, Dh=128, F=2048, axis_dims=(32, 48, 48),
                         pos_kind="3d", grid=(2, 10, 16), n_tail=22)
    inp = I.block_inputs(shape, seed=17, device=dev)
    cfg = h3lib.block_config(shape.S, shape.L, shape.D, shape.H, shape.Dh, shape.F,
                             shape.axis_dims, shape.theta, shape.eps_ln, shape.eps_qk)
    r = Guarded((shape.S, shape.D), torch.float32, fill=inp["resid"])
    nbytes = h3lib.block_workspace_bytes_fp8(cfg) if fp8 else h3lib.block_workspace_bytes(cfg)
    ws = Guarded((nbytes,), torch.uint8)
    if fp8:
        h3lib.block_forward_fp8(cfg, h3lib.quantize_block_weights_fp8(inp), r.t, inp["mod"],
                                inp["pos"], ws.t)
    else:
        h3lib.block_forward(cfg, inp, r.t, inp["mod"], inp["pos"], ws.t)
    h3lib.check_device_error()
    r.check("block resid")
    ws.check("block workspace")
    assert torch.equal(r.t[shape.L:], inp["resid"][shape.L:])
