"""The Python binding's tensor checks, on the CPU.

The C entry points take plain pointers, so the binding checks every tensor
before the call: element type, size, layout and residency on the handle's GPU.
Each case here builds tensors that are right in every respect but one and
expects TypeError / ValueError (never MxError, which would mean the C library
had been called). Tensors of the right type, size and layout that live in host
memory fail the last check, residency, so no pointer to host memory reaches a
kernel."""
import pytest
import torch


@pytest.fixture(scope="module")
def mx():
    import __graft_entry__

    __graft_entry__.build()
    import mxfp8_block_scaled_06_gb300 as mod

    mod.load_library()
    return mod


@pytest.fixture
def h(mx):
    return mx.Handle(0, 0)  # a null handle: any call that reached the library would fail there


def u8(*shape):
    return torch.zeros(shape, dtype=torch.uint8)


def bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def gemm_args(mx, m=4, n=256, k=512):
    return dict(a=u8(m, k), a_scales=u8(mx.mx_scale_bytes(m, k)), w=u8(n, k),
                w_scales=u8(mx.mx_scale_bytes(n, k)), out=bf16(m, n))


def test_host_tensors_fail_the_residency_check(mx, h):
    with pytest.raises(ValueError, match="cuda:0"):
        mx.mx_gemm(h, **gemm_args(mx))
    with pytest.raises(ValueError, match="cuda:0"):
        mx.mx_quantize_rows(h, bf16(4, 512))


@pytest.mark.parametrize("field,bad,exc,msg", [
    ("a", torch.zeros((4, 512), dtype=torch.float32), TypeError, "dtype"),
    ("a", u8(4, 256), ValueError, "shape"),
    ("a", u8(512, 4).t(), ValueError, "layout"),
    ("a_scales", u8(127 * 16), ValueError, "elements"),
    ("w", u8(256, 1024)[:, :512], ValueError, "layout"),
    ("w_scales", u8(10), ValueError, "elements"),
    ("out", bf16(4, 128), ValueError, "shape"),
    ("out", bf16(3, 256), ValueError, "shape"),
    ("out", torch.zeros((4, 256), dtype=torch.float16), TypeError, "dtype"),
])
def test_gemm_argument_checks(mx, h, field, bad, exc, msg):
    args = gemm_args(mx)
    args[field] = bad
    with pytest.raises(exc, match=msg):
        mx.mx_gemm(h, **args)


def test_gemm_rows_beyond_the_activation(mx, h):
    with pytest.raises(ValueError, match="shape"):
        mx.mx_gemm(h, **gemm_args(mx), m=5)


def test_float8_views_are_accepted_up_to_residency(mx, h):
    args = gemm_args(mx)
    args["a"] = args["a"].view(torch.float8_e4m3fn)
    args["w"] = args["w"].view(torch.float8_e4m3fn)
    with pytest.raises(ValueError, match="cuda:0"):
        mx.mx_gemm(h, **args)


def test_quantize_rows_checks(mx, h):
    with pytest.raises(ValueError, match="2-D"):
        mx.mx_quantize_rows(h, bf16(2, 4, 512))
    with pytest.raises(ValueError, match="layout"):
        mx.mx_quantize_rows(h, bf16(512, 4).t())
    with pytest.raises(ValueError, match="shape"):
        mx.mx_quantize_rows(h, bf16(4, 512), q=u8(4, 256))
    with pytest.raises(ValueError, match="elements"):  # plain scales: 4 x 16 bytes
        mx.mx_quantize_rows(h, bf16(4, 512), q=u8(4, 512), scales=u8(63), swizzled=False)
    with pytest.raises(ValueError, match="cuda:0"):  # a row-strided view is a valid layout
        mx.mx_quantize_rows(h, bf16(4, 640)[:, :512])


def test_chain_checks(mx, h):
    m = 2
    shapes = [(2048, 5120), (8192, 1536), (5120, 8192)]
    ws = [(u8(n, k), u8(mx.mx_scale_bytes(n, k))) for n, k in shapes]
    a1, a1s = u8(m, 5120), u8(mx.mx_scale_bytes(m, 5120))
    with pytest.raises(ValueError, match="three"):
        mx.mx_gemm_chain(h, a1, a1s, ws[:2])
    with pytest.raises(ValueError, match="shape"):
        mx.mx_gemm_chain(h, a1, a1s, ws, a2=u8(m, 1024))
    with pytest.raises(ValueError, match="elements"):
        mx.mx_gemm_chain(h, a1, a1s, ws, a3_scales=u8(100))
    with pytest.raises(ValueError, match="shape"):
        mx.mx_gemm_chain(h, u8(m, 4096), a1s, ws)
    with pytest.raises(ValueError, match="elements"):
        mx.mx_gemm_chain_norm(h, a1, a1s, ws, bf16(1024), 1e-6, a2=u8(m, 1536))
    with pytest.raises(ValueError, match="cuda:0"):
        mx.mx_gemm_chain_norm(h, a1, a1s, ws, bf16(1536), 1e-6)


def test_wo_a_checks(mx, h):
    G, H, R, D, t = 4, 8, 1024, 512, 3
    w, ws = u8(G * R, H * D), u8(mx.mx_scale_bytes(G * R, H * D))
    x, pos, cs = bf16(t, G * H, D), torch.zeros(t, dtype=torch.int64), torch.zeros((1024, 64))
    with pytest.raises(ValueError, match="contiguous elements"):
        mx.wo_a_grouped(h, bf16(t, G * H, D - 32), pos, cs, w, ws, G, H, R)
    with pytest.raises(ValueError, match="contiguous elements"):
        mx.wo_a_grouped(h, bf16(t, D, G * H).transpose(1, 2), pos, cs, w, ws, G, H, R)
    with pytest.raises(TypeError, match="dtype"):
        mx.wo_a_grouped(h, x, pos.int(), cs, w, ws, G, H, R)
    with pytest.raises(ValueError, match="elements"):
        mx.wo_a_grouped(h, x, pos[:2], cs, w, ws, G, H, R)
    with pytest.raises(ValueError, match="max_pos"):
        mx.wo_a_grouped(h, x, pos, torch.zeros((1024, 32)), w, ws, G, H, R)
    with pytest.raises(ValueError, match="shape"):
        mx.wo_a_grouped_unfused(h, x, pos, cs, w, ws, G, H, R, xq=u8(t, 1024))
    with pytest.raises(ValueError, match="cuda:0"):  # tokens strided inside a wider buffer
        mx.wo_a_grouped(h, bf16(t, 2 * G * H, D)[:, :G * H], pos, cs, w, ws, G, H, R)


def test_python_scale_size_matches_the_library(mx):
    for rows in (0, 1, 5, 127, 128, 129, 300):
        for k in (0, 16, 32, 96, 128, 160, 5120, 8200):
            assert mx._sbytes(rows, k) == mx.mx_scale_bytes(rows, k), (rows, k)


def test_unpinned_host_memory_is_refused_where_pinned_is_accepted(mx, h):
    # x of mx_quantize_rows and out of mx_gemm may be pinned host memory; a plain
    # (pageable) host tensor is still refused before any call
    with pytest.raises(ValueError, match="pinned host memory"):
        mx.mx_quantize_rows(h, bf16(4, 512))
    args = gemm_args(mx)
    with pytest.raises(ValueError, match="cuda:0"):
        mx.mx_gemm(h, **args)
