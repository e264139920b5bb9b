"""Guard canaries around every output of every entry point.

Each output is a view into a larger device buffer whose leading and trailing
bytes hold a known pattern; after the call the guards must be intact, so a
kernel writing past either end of an output (wrong index arithmetic, padding
beyond the documented size) fails here, on shapes with ragged rows and tiles.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import bf16_to_device, handle, quantize_on_gpu

pytestmark = pytest.mark.gpu

PAD = 4096          # guard bytes on each side (keeps 16-byte alignment)
PATTERN = 0xA5


class Guarded:
    def __init__(self):
        self.bufs = []

    def u8(self, nbytes):
        buf = torch.full((nbytes + 2 * PAD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.bufs.append((buf, nbytes))
        return buf[PAD:PAD + nbytes]

    def bf16(self, rows, cols):
        return self.u8(rows * cols * 2).view(torch.bfloat16).view(rows, cols)

    def check(self):
        torch.cuda.synchronize()
        for buf, n in self.bufs:
            host = buf.cpu().numpy()
            assert (host[:PAD] == PATTERN).all(), "write before the start of an output"
            assert (host[PAD + n:] == PATTERN).all(), "write past the end of an output"


@pytest.mark.parametrize("m,k", [(1, 64), (5, 160), (130, 96), (3, 5120)])
def test_quantize_rows_guards(m, k):
    import mxfp8_block_scaled_06_gb300 as mx

    g = Guarded()
    x = bf16_to_device(synth.block_scaled_bf16(1, synth.TAG_A, m, k, -6, 6))
    q = g.u8(m * k).view(m, k)
    s = g.u8(mx.mx_scale_bytes(m, k))
    mx.mx_quantize_rows(handle(), x, q=q, scales=s)
    q2 = g.u8(m * k).view(m, k)
    s2 = g.u8(m * (k // 32))
    mx.mx_quantize_rows(handle(), x, q=q2, scales=s2, swizzled=False)
    g.check()


@pytest.mark.parametrize("m,n,k", [(1, 2048, 5120), (17, 384, 640), (130, 256, 512), (64, 8192, 1536)])
def test_gemm_and_bf16_gemm_guards(m, n, k):
    import mxfp8_block_scaled_06_gb300 as mx

    g = Guarded()
    abits = synth.block_scaled_bf16(2, synth.TAG_A, m, k, -6, 6)
    aq, asc = quantize_on_gpu(abits)
    wq, wsc = quantize_on_gpu(synth.block_scaled_bf16(2, synth.TAG_W, n, k, -6, 6))
    out = g.bf16(m, n)
    mx.mx_gemm(handle(), aq, asc, wq, wsc, out=out, pdl=True)
    out2 = g.bf16(m, n)
    mx.mx_gemm_bf16(handle(), bf16_to_device(abits), wq, wsc, out=out2)
    g.check()
    assert mx.mx_device_status(handle()) == mx.MX_OK


@pytest.mark.parametrize("m", [1, 17])
def test_chain_guards(m):
    import mxfp8_block_scaled_06_gb300 as mx

    g = Guarded()
    shapes = [(2048, 5120), (8192, 1536), (5120, 8192)]
    ws = [quantize_on_gpu(synth.block_scaled_bf16(3 + i, synth.TAG_W, n, k, -6, 6))
          for i, (n, k) in enumerate(shapes)]
    a1 = quantize_on_gpu(synth.block_scaled_bf16(3, synth.TAG_A, m, 5120, -4, 4))
    bufs = dict(out=g.bf16(m, 5120),
                a2=g.u8(m * 1536).view(m, 1536), a2_scales=g.u8(mx.mx_scale_bytes(m, 1536)),
                a3=g.u8(m * 8192).view(m, 8192), a3_scales=g.u8(mx.mx_scale_bytes(m, 8192)))
    mx.mx_gemm_chain(handle(), a1[0], a1[1], ws, **bufs)
    g.check()
    assert mx.mx_device_status(handle()) == mx.MX_OK


@pytest.mark.parametrize("t", [1, 9, 33])
def test_wo_a_guards(t):
    import mxfp8_block_scaled_06_gb300 as mx

    G, H, R, D = 4, 8, 1024, 512
    g = Guarded()
    ww = quantize_on_gpu(synth.block_scaled_bf16(4, synth.TAG_WOA, G * R, H * D, -6, 6))
    cs = torch.from_numpy(synth.rope_cos_sin_cache(65536)).cuda()
    x = bf16_to_device(synth.normal_bf16(4, synth.TAG_X, (t, G * H, D)))
    pos = torch.from_numpy(synth.positions(4, synth.TAG_POS, t)).cuda()
    q = g.u8(t * G * R).view(t, G * R)
    qs = g.u8(mx.mx_scale_bytes(t, G * R))
    mx.wo_a_grouped(handle(), x, pos, cs, *ww, G, H, R, q=q, q_scales=qs)
    q2 = g.u8(t * G * R).view(t, G * R)
    qs2 = g.u8(mx.mx_scale_bytes(t, G * R))
    xq = g.u8(t * G * H * D).view(t, G * H * D)
    xqs = g.u8(mx.mx_scale_bytes(t, G * H * D))
    mx.wo_a_grouped_unfused(handle(), x, pos, cs, *ww, G, H, R, q=q2, q_scales=qs2, xq=xq,
                            xq_scales=xqs)
    g.check()
    assert mx.mx_device_status(handle()) == mx.MX_OK


def test_empty_inputs_are_rejected_and_launch_nothing():
    """Zero rows or tokens: every entry point returns MX_ERR_INVALID_ARG before
    any launch (the documented domain starts at one row), and no output byte
    changes."""
    import mxfp8_block_scaled_06_gb300 as mx

    lib, h = mx.load_library(), handle().ptr
    g = Guarded()
    k, n = 512, 256
    x = bf16_to_device(synth.block_scaled_bf16(6, synth.TAG_A, 4, k, -4, 4))
    nw = torch.ones(k, dtype=torch.bfloat16, device="cuda")
    wq, wsc = quantize_on_gpu(synth.block_scaled_bf16(6, synth.TAG_W, n, k, -6, 6))
    aq, asc = quantize_on_gpu(synth.block_scaled_bf16(6, synth.TAG_A, 4, k, -6, 6))
    q, s, out = g.u8(4 * k), g.u8(mx.mx_scale_bytes(4, k)), g.u8(4 * n * 2)
    p = lambda t: t.data_ptr()
    err = mx.MX_ERR_INVALID_ARG
    assert lib.mx_quantize_rows(h, 0, k, p(x), k, p(q), p(s), 1, None) == err
    assert lib.mx_rmsnorm_quantize_rows(h, 0, k, p(x), k, p(nw), 1e-6, None, p(q), p(s), 1, None) == err
    assert lib.mx_gemm(h, 0, n, k, p(aq), p(asc), p(wq), p(wsc), p(out), 0, None) == err
    assert lib.mx_gemm_bf16(h, 0, n, k, p(x), k, p(wq), p(wsc), p(out), 0, None) == err
    # three [256, 512] weights: the row count is checked first
    ws = (mx.MxWeight * 3)(*[mx.MxWeight(p(wq), p(wsc), n, k)] * 3)
    assert lib.mx_gemm_chain(h, 0, p(aq), p(asc), ws, 512, p(q), p(s), p(q), p(s), p(out),
                             None, None, None) == err
    assert lib.mx_gemm_chain_norm(h, 0, p(aq), p(asc), ws, 512, p(nw), 1e-6, p(out), p(q), p(s),
                                  p(q), p(s), p(out), None, None, None) == err
    G, H, R, D = 4, 8, 1024, 512
    ww = quantize_on_gpu(synth.block_scaled_bf16(6, synth.TAG_WOA, G * R, H * D, -6, 6))
    cs = torch.zeros((16, 64), dtype=torch.float32, device="cuda")
    xt = torch.zeros((1, G * H, D), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(1, dtype=torch.int64, device="cuda")
    assert lib.wo_a_grouped(h, 0, p(xt), G * H * D, p(pos), p(cs), 16, p(ww[0]), p(ww[1]), G, H, 448,
                            64, R, p(q), p(s), None, None, None, 0, None) == err
    assert lib.wo_a_grouped_unfused(h, 0, p(xt), G * H * D, p(pos), p(cs), 16, p(ww[0]), p(ww[1]), G,
                                    H, 448, 64, R, p(q), p(s), None, p(q), p(s), None) == err
    g.check()
    for buf, nbytes in g.bufs:  # the outputs themselves are untouched too
        assert (buf[PAD:PAD + nbytes].cpu().numpy() == PATTERN).all()
    assert mx.mx_device_status(handle()) == mx.MX_OK


@pytest.mark.parametrize("fault", ["n_not_tiled", "k_mismatch", "scales_misaligned"])
def test_chain_rejecting_its_third_projection_writes_nothing(fault):
    """A chain whose third projection is rejected fails before its first launch:
    out1 / out2, a2, a3 and out keep every byte (the cute_dsl page's `_consumer`
    validates before any launch). Called through the C ABI, so the binding's own
    checks do not stand in front of the library's."""
    import mxfp8_block_scaled_06_gb300 as mx

    lib, h = mx.load_library(), handle().ptr
    m, (n1, k1), (n2, k2), (n3, k3) = 4, (384, 640), (256, 256), (512, 256)
    w = [quantize_on_gpu(synth.block_scaled_bf16(7 + i, synth.TAG_W, n, k, -6, 6))
         for i, (n, k) in enumerate([(n1, k1), (n2, k2), (n3, k3)])]
    aq, asc = quantize_on_gpu(synth.block_scaled_bf16(7, synth.TAG_A, m, k1, -4, 4))
    nw = torch.ones(k2, dtype=torch.bfloat16, device="cuda")
    p = lambda t: t.data_ptr()
    third = {"n_not_tiled": (p(w[2][0]), p(w[2][1]), n3 + 64, k3, mx.MX_ERR_UNSUPPORTED),
             "k_mismatch": (p(w[2][0]), p(w[2][1]), n3, k3 + 128, mx.MX_ERR_INVALID_ARG),
             "scales_misaligned": (p(w[2][0]), p(w[2][1]) + 16, n3, k3, mx.MX_ERR_INVALID_ARG)}[fault]
    ws = (mx.MxWeight * 3)(mx.MxWeight(p(w[0][0]), p(w[0][1]), n1, k1),
                           mx.MxWeight(p(w[1][0]), p(w[1][1]), n2, k2),
                           mx.MxWeight(*third[:4]))
    g = Guarded()
    out1, out2, out = g.u8(m * n1 * 2), g.u8(m * n2 * 2), g.u8(m * (n3 + 64) * 2)
    a2, a2s = g.u8(m * k2), g.u8(mx.mx_scale_bytes(m, k2))
    a3, a3s = g.u8(m * n2), g.u8(mx.mx_scale_bytes(m, n2))
    y = g.u8(m * k2 * 2)
    torch.cuda.synchronize()
    assert lib.mx_gemm_chain(h, m, p(aq), p(asc), ws, k2, p(a2), p(a2s), p(a3), p(a3s), p(out),
                             p(out1), p(out2), None) == third[4]
    assert lib.mx_gemm_chain_norm(h, m, p(aq), p(asc), ws, k2, p(nw), 1e-6, p(out1), p(a2), p(a2s),
                                  p(a3), p(a3s), p(out), p(y), p(out2), None) == third[4]
    g.check()
    for buf, nbytes in g.bufs:
        assert (buf[PAD:PAD + nbytes].cpu().numpy() == PATTERN).all(), "a rejected chain wrote an output"
    assert mx.mx_device_status(handle()) == mx.MX_OK
