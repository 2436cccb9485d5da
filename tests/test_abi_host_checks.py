"""Host-side argument checks of the device-facing C-ABI calls, on the CPU.

Every device call validates its views and arguments before it touches the
CUDA runtime, so malformed calls are refused with a status code and a
message on a machine without a GPU.  The views here carry fake, aligned
device addresses that are never dereferenced; only calls that must fail are
made, so nothing is ever launched."""
import ctypes

import pytest

from decode_gemv_gb300 import lw

FAKE = 0x7F0000000000          # 16-byte aligned, never dereferenced


def view(fmt=lw.LW_FMT_Q4_PAIR, twin=0, rows=128, cols=512, max_tile_rows=40, lmin=3, lmax=9, base=FAKE):
    v = lw.LwDevBundle()
    v.fmt, v.twin, v.rows, v.cols = fmt, twin, rows, cols
    v.max_tile_rows, v.lmin, v.lmax = max_tile_rows, lmin, lmax
    for i, name in enumerate(lw.SECTION_NAMES):
        setattr(v, name, base + 0x100000 * (i + 1))
    if twin:
        v.lane_mid = None
    return v


def P(x):
    return ctypes.c_void_p(x)


@pytest.fixture(scope="module")
def lib():
    # the views carry fake device addresses: never let a call that could
    # launch run where a GPU is visible
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("host-check tests run only where no GPU is visible")
    return lw.load()


def status(lib, fn, *args):
    st = getattr(lib, fn)(*args)
    msg = lib.lw_last_error().decode()
    return st, msg


def test_product_argument_errors(lib):
    v = view()
    ws, x, y = P(FAKE + 0x9000000), P(FAKE + 0xA000000), P(FAKE + 0xB000000)
    need = lib.lw_workspace_bytes(ctypes.byref(v), 1)
    assert need > 0
    cases = [
        (ctypes.byref(view(fmt=9)), 1, ws, need, lw.LW_ERR_UNSUPPORTED),
        (ctypes.byref(view(rows=100)), 1, ws, need, lw.LW_ERR_SHAPE),
        (ctypes.byref(view(cols=300)), 1, ws, need, lw.LW_ERR_SHAPE),
        (ctypes.byref(v), 0, ws, need, lw.LW_ERR_INVALID_ARG),           # batch 0
        (ctypes.byref(v), 257, ws, 1 << 40, lw.LW_ERR_INVALID_ARG),      # batch 257
        (ctypes.byref(v), 1, None, need, lw.LW_ERR_INVALID_ARG),         # no workspace
        (ctypes.byref(v), 1, ws, need - 4, lw.LW_ERR_INVALID_ARG),       # too small
        (ctypes.byref(v), 1, P(FAKE + 8), need, lw.LW_ERR_INVALID_ARG),  # misaligned
        (ctypes.byref(view(twin=1)), 1, ws, need, lw.LW_ERR_INVALID_ARG),   # twin to the coded call
        (ctypes.byref(view(lmin=0)), 1, ws, need, lw.LW_ERR_INVALID_ARG),
        (ctypes.byref(view(max_tile_rows=5000)), 1, ws, need, lw.LW_ERR_INVALID_ARG),
    ]
    for vb, batch, w, wb, want in cases:
        st, msg = status(lib, "lw_decode_gemm", vb, x, batch, y, w, wb, None, None)
        assert st == want, (st, want, msg)
        assert msg
    v2 = view()
    v2.lane_mid = None
    st, msg = status(lib, "lw_decode_gemv", ctypes.byref(v2), x, y, ws, need, None, None)
    assert st == lw.LW_ERR_INVALID_ARG and msg
    # the twin call refuses a coded bundle
    st, msg = status(lib, "lw_twin_gemv", ctypes.byref(v), x, y, ws, need, None, None)
    assert st == lw.LW_ERR_INVALID_ARG and msg


def test_group_argument_errors(lib):
    vs = [view(), view(rows=256), view(fmt=lw.LW_FMT_Q6), view(fmt=lw.LW_FMT_BF16_EXP), view(twin=1)]
    arr = lambda idx: (ctypes.c_void_p * len(idx))(*[ctypes.addressof(vs[i]) for i in idx])
    ptrs = lambda n, off: (ctypes.c_void_p * max(n, 1))(*[FAKE + off + 0x100000 * i for i in range(max(n, 1))])
    ws = P(FAKE + 0x9000000)
    need = lib.lw_workspace_bytes_group(arr([0, 1]), 2)
    assert need >= lib.lw_workspace_bytes(ctypes.byref(vs[0]), 1) + lib.lw_workspace_bytes(ctypes.byref(vs[1]), 1)
    assert lib.lw_workspace_bytes_group(arr([0]), 0) == 0
    assert lib.lw_workspace_bytes_group(arr([0] * 9), 9) == 0
    cases = [
        ("lw_decode_gemv_group", [0], 0, need, lw.LW_ERR_INVALID_ARG),          # n = 0
        ("lw_decode_gemv_group", [0] * 9, 9, 1 << 40, lw.LW_ERR_INVALID_ARG),  # n = 9
        ("lw_decode_gemv_group", [0, 2], 2, 1 << 40, lw.LW_ERR_INVALID_ARG),   # mixed formats
        ("lw_decode_gemv_group", [3], 1, 1 << 40, lw.LW_ERR_UNSUPPORTED),      # BF16
        ("lw_decode_gemv_group", [0, 4], 2, 1 << 40, lw.LW_ERR_INVALID_ARG),   # a twin
        ("lw_decode_gemv_group", [0, 1], 2, need - 16, lw.LW_ERR_INVALID_ARG),  # workspace
        ("lw_twin_gemv_group", [0], 1, 1 << 40, lw.LW_ERR_INVALID_ARG),        # a coded bundle
    ]
    for fn, idx, n, wb, want in cases:
        st, msg = status(lib, fn, arr(idx), n, ptrs(len(idx), 0xA000000), ptrs(len(idx), 0xB000000),
                         ws, wb, None, None)
        assert st == want, (fn, idx, st, want, msg)
        assert msg
    # a misaligned activation pointer
    xs = ptrs(2, 0xA000000)
    xs[1] = FAKE + 0xA000004
    st, msg = status(lib, "lw_decode_gemv_group", arr([0, 1]), 2, xs, ptrs(2, 0xB000000), ws, 1 << 40,
                     None, None)
    assert st == lw.LW_ERR_INVALID_ARG and msg


def test_strip_list_argument_errors(lib):
    v = view()
    x, y, ws = P(FAKE + 0xA000000), P(FAKE + 0xB000000), P(FAKE + 0x9000000)
    s = P(FAKE + 0xC000000)
    need = lib.lw_workspace_bytes(ctypes.byref(v), 1)
    cases = [
        (ctypes.byref(view(fmt=lw.LW_FMT_BF16_EXP)), s, 1, need, lw.LW_ERR_UNSUPPORTED),
        (ctypes.byref(view(twin=1)), s, 1, need, lw.LW_ERR_INVALID_ARG),
        (ctypes.byref(v), s, 3, need, lw.LW_ERR_INVALID_ARG),           # 3 > 128 / 64 strips
        (ctypes.byref(v), None, 1, need, lw.LW_ERR_INVALID_ARG),        # no list
        (ctypes.byref(v), s, -1, need, lw.LW_ERR_INVALID_ARG),
        (ctypes.byref(v), P(FAKE + 0xC000002), 1, need, lw.LW_ERR_INVALID_ARG),   # misaligned list
        (ctypes.byref(v), s, 1, 16, lw.LW_ERR_INVALID_ARG),             # workspace
    ]
    for vb, lst, n, wb, want in cases:
        st, msg = status(lib, "lw_decode_gemm_strips", vb, lst, n, x, 1, y, ws, wb, None, None)
        assert st == want, (n, st, want, msg)
        assert msg
    # an empty list launches nothing and succeeds
    st, _ = status(lib, "lw_decode_gemm_strips", ctypes.byref(v), None, 0, x, 1, y, ws, need, None, None)
    assert st == lw.LW_OK


def test_transcode_argument_errors(lib):
    coded = view()
    tw = view(twin=1, max_tile_rows=lib.lw_twin_tile_rows(lw.LW_FMT_Q4_PAIR), base=FAKE + 0x40000000)
    assert lib.lw_twin_tile_rows(lw.LW_FMT_Q4_PAIR) == 64
    assert lib.lw_twin_tile_rows(lw.LW_FMT_Q6) == 96
    assert lib.lw_twin_tile_rows(lw.LW_FMT_BF16_EXP) == 64
    assert lib.lw_twin_tile_rows(0) == 0
    def bad(**kw):
        t = view(twin=1, max_tile_rows=64, base=FAKE + 0x40000000)
        for k, val in kw.items():
            setattr(t, k, val)
        return t
    cases = [
        (view(twin=1), tw),                      # a twin as the source
        (coded, bad(twin=0)),
        (coded, bad(fmt=lw.LW_FMT_Q6)),
        (coded, bad(rows=256)),
        (coded, bad(max_tile_rows=63)),
        (coded, bad(words=None)),
        (coded, bad(words=FAKE + 0x40000008)),   # misaligned
        (coded, bad(words=coded.words)),         # on top of the coded words
        (coded, bad(words=coded.lane_mid - 64)),  # overlapping the lane mids
    ]
    for c, t in cases:
        st, msg = status(lib, "lw_transcode_twin", ctypes.byref(c), ctypes.byref(t), None, None)
        assert st == lw.LW_ERR_INVALID_ARG, (st, msg)
        assert msg


def test_gemm_group_batch_checks(lib):
    vs = [view(), view(rows=256)]
    arr = (ctypes.c_void_p * 2)(*[ctypes.addressof(v) for v in vs])
    xs = (ctypes.c_void_p * 2)(FAKE + 0xA000000, FAKE + 0xA100000)
    ys = (ctypes.c_void_p * 2)(FAKE + 0xB000000, FAKE + 0xB100000)
    ws = P(FAKE + 0x9000000)
    for fn in ("lw_decode_gemm_group", "lw_twin_gemm_group"):
        for batch in (0, 9, -1):
            st, msg = status(lib, fn, arr, 2, xs, batch, ys, ws, 1 << 40, None, None)
            assert st == lw.LW_ERR_INVALID_ARG and msg, (fn, batch, st)


def test_stall_hook_arguments(lib):
    """The testing hook checks its range; 0 withdraws a pending request (so
    this test leaves none behind)."""
    for bad in (-1, 1000001):
        st, msg = status(lib, "lw_test_stall_next", bad)
        assert st == 1 and "wait_us" in msg
    assert lib.lw_test_stall_next(5) == 0
    assert lib.lw_test_stall_next(0) == 0


def test_no_alloc_argument_errors(lib):
    """lw_decode_gemv_noalloc checks its arguments before it queues anything:
    on a machine without a GPU the refusals name the argument (a queued clear
    of the shared counters would fail first with LW_ERR_CUDA)."""
    v = view()
    x, y = P(FAKE + 0xA000000), P(FAKE + 0xB000000)
    cases = [
        (ctypes.byref(view(fmt=9)), x, y, lw.LW_ERR_UNSUPPORTED),
        (ctypes.byref(view(rows=100)), x, y, lw.LW_ERR_SHAPE),
        (ctypes.byref(v), None, y, lw.LW_ERR_INVALID_ARG),
        (ctypes.byref(v), x, None, lw.LW_ERR_INVALID_ARG),
        (ctypes.byref(v), P(FAKE + 0xA000008), y, lw.LW_ERR_INVALID_ARG),   # x misaligned
        (ctypes.byref(v), x, P(FAKE + 0xB000004), lw.LW_ERR_INVALID_ARG),   # y misaligned
        (ctypes.byref(view(twin=1)), x, y, lw.LW_ERR_INVALID_ARG),
    ]
    for vb, xx, yy, want in cases:
        st, msg = status(lib, "lw_decode_gemv_noalloc", vb, xx, yy, None, None)
        assert st == want, (st, want, msg)
        assert "clearing" not in msg
    # a matrix beyond the scratch is refused before any device work
    big = view(rows=64 * 1024, cols=256 * 64)
    st, msg = status(lib, "lw_decode_gemv_noalloc", ctypes.byref(big), x, y, None, None)
    assert st == lw.LW_ERR_UNSUPPORTED and "scratch" in msg
