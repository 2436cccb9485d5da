"""The Python binding checks every tensor before its address reaches the C
ABI: a tensor of the wrong dtype, strided, too small for the view's shape or
on the host is refused with LW_ERR_INVALID_ARG and nothing is called.

Runs on the CPU: the bundles are encoded by the library's host code and
"uploaded" to host tensors, and the library handle is swapped for a guard
that fails the test if any device call is reached."""
import numpy as np
import pytest

from decode_gemv_gb300 import inputs
from decode_gemv_gb300 import lw

torch = pytest.importorskip("torch")


class _Guard:
    """Stands in for the loaded library: any call through it is a failure."""

    def __getattr__(self, name):
        raise AssertionError(f"{name} was called although the binding should have refused")


@pytest.fixture
def q4():
    m = inputs.small_q4(3, 128, 512)
    hb = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m["codes"], m["scales"], m["mins"])
    return lw.DeviceBundle.upload(hb, "cpu")


@pytest.fixture
def q6():
    m = inputs.small_q6(4, 64, 256)
    hb = lw.lw_encode_bundle(lw.LW_FMT_Q6, m["codes"], m["scales"])
    return lw.DeviceBundle.upload(hb, "cpu")


@pytest.fixture
def bf16():
    m = inputs.small_bf16(5, 64, 256)
    hb = lw.lw_encode_bundle(lw.LW_FMT_BF16_EXP, m["bits"])
    return lw.DeviceBundle.upload(hb, "cpu")


@pytest.fixture
def guarded(monkeypatch):
    lw.load()
    monkeypatch.setattr(lw, "_lib", _Guard())


def _refused(call, *words):
    with pytest.raises(lw.LwError) as e:
        call()
    assert e.value.status == lw.LW_ERR_INVALID_ARG
    for w in words:
        assert w in str(e.value), str(e.value)


def f32(n):
    return torch.zeros(n, dtype=torch.float32)


def i32(n=1):
    return torch.zeros(n, dtype=torch.int32)


def test_gemv_activation_and_output_checks(q4, guarded):
    N, K = q4.rows, q4.cols
    ws = f32(1 << 12)
    call = lambda x, y: lw.lw_decode_gemv(q4, x, y, ws, i32())
    _refused(lambda: call(np.zeros(K, np.float32), f32(N)), "x:", "torch.Tensor")
    _refused(lambda: call(torch.zeros(K, dtype=torch.float64), f32(N)), "x:", "dtype float64")
    _refused(lambda: call(f32(2 * K)[::2], f32(N)), "x:", "not contiguous")
    _refused(lambda: call(f32(K - 1), f32(N)), "x:", f"{4 * (K - 1)} bytes", f"needs {4 * K}")
    _refused(lambda: call(f32(K), torch.zeros(N, dtype=torch.float16)), "y:", "dtype float16")
    _refused(lambda: call(f32(K), f32(N - 64)), "y:", f"needs {4 * N}")
    # every buffer is well formed: the devices are checked next, the
    # bundle's first
    for fn in (lw.lw_twin_gemv, lw.lw_decode_gemv):
        _refused(lambda fn=fn: fn(q4, f32(K), f32(N), ws, i32()), "bundle:", "sections on cpu")
    _refused(lambda: lw.lw_decode_gemv_noalloc(q4, f32(K - 4), f32(N), i32()), "x:", "bytes")


def test_gemm_sizes_follow_the_batch(q6, guarded):
    N, K, B = q6.rows, q6.cols, 3
    ws = f32(1 << 12)
    _refused(lambda: lw.lw_decode_gemm(q6, f32(B * K - 1), B, f32(B * N), ws, i32()),
             "X:", f"needs {4 * B * K}")
    _refused(lambda: lw.lw_twin_gemm(q6, f32(B * K), B, f32(B * N - 1), ws, i32()),
             "Y:", f"needs {4 * B * N}")
    _refused(lambda: lw.lw_decode_gemm(q6, f32(B * K).view(B, K).t(), B, f32(B * N), ws, i32()),
             "X:", "not contiguous")
    _refused(lambda: lw.lw_decode_gemm(q6, f32(B * K), B, f32(B * N), ws, i32()), "sections on cpu")


def test_bf16_activations_are_two_byte(bf16, guarded):
    N, K = bf16.rows, bf16.cols
    ws = f32(1 << 12)
    _refused(lambda: lw.lw_decode_gemv(bf16, f32(K), f32(N), ws, i32()), "x:", "dtype float32",
             "bfloat16")
    _refused(lambda: lw.lw_decode_gemv(bf16, torch.zeros(K - 1, dtype=torch.bfloat16), f32(N),
                                       ws, i32()), f"needs {2 * K}")
    for dt in (torch.bfloat16, torch.int16):      # the value or its bits
        _refused(lambda dt=dt: lw.lw_decode_gemv(bf16, torch.zeros(K, dtype=dt), f32(N), ws, i32()),
                 "bundle:", "sections on cpu")


def test_decode_output_size_per_format(q4, q6, bf16, guarded):
    for db, per_weight in ((q4, 0.5), (q6, 1), (bf16, 2)):
        need = int(db.rows * db.cols * per_weight)
        _refused(lambda db=db, need=need: lw.lw_decode(db, torch.zeros(need - 1, dtype=torch.uint8),
                                                       i32()), "out:", f"needs {need}")
        _refused(lambda db=db, need=need: lw.lw_decode(db, torch.zeros(need, dtype=torch.uint8),
                                                       i32()), "sections on cpu")


def test_status_and_strip_list_types(q4, guarded):
    N, K = q4.rows, q4.cols
    _refused(lambda: lw.lw_decode_gemm_strips(q4, torch.zeros(1, dtype=torch.int64), f32(K), 1,
                                              f32(N), f32(1 << 12), i32()), "strips:", "int64")
    _refused(lambda: lw.lw_decode_gemm_strips(q4, i32(2)[:1].expand(3), f32(K), 1, f32(N),
                                              f32(1 << 12), i32()), "strips:")
    # the device status: one int32
    _refused(lambda: lw.lw_decode_gemv(q4, f32(K), f32(N), f32(16), torch.zeros(1, dtype=torch.int64)),
             "d_status:", "int64")
    _refused(lambda: lw.lw_decode(q4, torch.zeros(N * K // 2, dtype=torch.uint8), i32(0)),
             "d_status:", "0 bytes")


def test_buffers_must_be_on_the_bundles_device():
    cuda0, cuda1 = torch.device("cuda", 0), torch.device("cuda", 1)
    _refused(lambda: lw._on("call", cuda0, ("y", f32(4))), "y: on cpu, expected a CUDA device")
    _refused(lambda: lw._on("call", cuda1, ("x", torch.empty(4, device="meta"))), "x: on meta")


def test_groups_check_every_member(q4, guarded):
    N, K = q4.rows, q4.cols
    ws = f32(1 << 12)
    _refused(lambda: lw.lw_decode_gemv_group([q4, q4], [f32(K)], [f32(N), f32(N)], ws, i32()),
             "2 bundles, 1 activations")
    _refused(lambda: lw.lw_decode_gemv_group([q4, q4], [f32(K), f32(K)], [f32(N), f32(N - 1)],
                                             ws, i32()), "y[1]:", "bytes")
    _refused(lambda: lw.lw_twin_gemm_group([q4, q4], [f32(2 * K), f32(K)], 2, [f32(2 * N)] * 2,
                                           ws, i32()), "x[1]:", f"needs {8 * K}")
    _refused(lambda: lw.PreparedGemv([q4], [f32(K)], [f32(N)], ws, i32()), "bundle[0]:",
             "sections on cpu")
    _refused(lambda: lw.PreparedGemv([q4], [f32(K)], [f32(N - 1)], ws, i32()), "y[0]:", "bytes")
    _refused(lambda: lw.PreparedGemv([q4, q4], [f32(K)] * 2, [f32(N)], ws, i32()),
             "2 bundles, 2 activations, 1 outputs")


def test_bundle_must_sit_on_one_cuda_device(q4):
    with pytest.raises(lw.LwError) as e:
        lw._bundle_device("call", q4)
    assert e.value.status == lw.LW_ERR_INVALID_ARG and "sections on cpu" in str(e.value)


def test_shapes_the_library_refuses_are_left_to_it(q4):
    """A view whose shape the C call rejects (LW_ERR_SHAPE) needs no buffer
    size: the binding does not pre-empt the library's own status."""
    assert lw._dims(q4) == (q4.rows, q4.cols)
    q4.view.rows = 65
    assert lw._dims(q4) == (0, 0)
    q4.view.rows, q4.view.cols = 64, 300
    assert lw._dims(q4) == (0, 0)
