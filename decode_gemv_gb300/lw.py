"""Thin Python binding of liblw (the C ABI in include/lw.h).

Argument marshalling and checks only: every step of the path runs in liblw's
host code or CUDA kernels.  Each tensor is checked (dtype, contiguity, size,
device) before its address crosses the ABI, since the C calls cannot see
them.  PyTorch is used for device memory and streams.  If the compiled
library is missing this module raises at load time -- there is no fallback.
Functions carry the C names; see include/lw.h for the contract of each.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "liblw.so")

LW_FMT_Q4_PAIR, LW_FMT_Q6, LW_FMT_BF16_EXP = 1, 2, 3
# device status codes (*d_status), as in include/lw.h
(LW_DEV_OK, LW_DEV_LANE_LENGTH, LW_DEV_BAD_CODE, LW_DEV_TILE_SIZE, LW_DEV_TIMEOUT,
 LW_DEV_BAD_TABLE, LW_DEV_BAD_STRIPS) = range(7)
(LW_OK, LW_ERR_INVALID_ARG, LW_ERR_SHAPE, LW_ERR_UNSUPPORTED, LW_ERR_ALLOC, LW_ERR_CORRUPT,
 LW_ERR_CUDA, LW_ERR_IO) = range(8)
SECTION_NAMES = ["words", "tile_off", "lane_bits", "table", "qparams", "signman",
                 "vflags", "vrow_off", "vexp", "lane_mid"]
STATUS_NAMES = {0: "LW_OK", 1: "LW_ERR_INVALID_ARG", 2: "LW_ERR_SHAPE", 3: "LW_ERR_UNSUPPORTED",
                4: "LW_ERR_ALLOC", 5: "LW_ERR_CORRUPT", 6: "LW_ERR_CUDA", 7: "LW_ERR_IO"}
DEV_STATUS = {0: "ok", 1: "lane length", 2: "bad code", 3: "tile size", 4: "timeout",
              5: "bad table"}
TABLE_BYTES = 1024
EXPORTED = ["lw_encode_bundle", "lw_bundle_sections", "lw_bundle_free", "lw_table_from_lengths",
            "lw_validate_sections", "lw_workspace_bytes", "lw_decode", "lw_decode_gemv",
            "lw_decode_gemm", "lw_twin_gemv", "lw_twin_gemm", "lw_status_string",
            "lw_last_error", "lw_version", "lw_decode_gemv_noalloc", "lw_noalloc_scratch_bytes",
            "lw_decode_gemv_group", "lw_workspace_bytes_group", "lw_twin_gemv_group",
            "lw_bundle_desc", "lw_bundle_serialized_bytes", "lw_bundle_serialize",
            "lw_bundle_deserialize", "lw_bundle_save", "lw_bundle_load", "lw_transcode_twin",
            "lw_twin_tile_rows", "lw_decode_gemm_strips", "lw_graph_begin", "lw_graph_end",
            "lw_graph_launch", "lw_graph_free", "lw_decode_gemm_group", "lw_twin_gemm_group",
            "lw_table_lut_entries", "lw_test_stall_next"]


class LwError(RuntimeError):
    """A failing call: `status` is the lw_status code.  `detail` replaces the
    library's thread-local error text when the binding itself refused the
    call before reaching the library."""

    def __init__(self, status: int, what: str, detail: str | None = None):
        self.status = status
        text = _last_error() if detail is None else detail
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}: {text}")


class LwDesc(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("twin", ctypes.c_int32),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


class LwSections(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p * 10), ("bytes", ctypes.c_uint64 * 10),
                ("coded_bytes", ctypes.c_uint64), ("n_tiles", ctypes.c_uint64),
                ("n_verbatim", ctypes.c_int64), ("max_tile_rows", ctypes.c_int32),
                ("max_len", ctypes.c_int32), ("min_len", ctypes.c_int32),
                ("palette_size", ctypes.c_int32), ("bits_per_weight", ctypes.c_double),
                ("lut_entries", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class LwDevBundle(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("twin", ctypes.c_int32),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("max_tile_rows", ctypes.c_int32), ("lmin", ctypes.c_int32),
                ("lmax", ctypes.c_int32), ("lut_entries", ctypes.c_int32),
                ("words", ctypes.c_void_p), ("tile_off", ctypes.c_void_p),
                ("lane_bits", ctypes.c_void_p), ("table", ctypes.c_void_p),
                ("qparams", ctypes.c_void_p), ("signman", ctypes.c_void_p),
                ("vflags", ctypes.c_void_p), ("vrow_off", ctypes.c_void_p),
                ("vexp", ctypes.c_void_p), ("lane_mid", ctypes.c_void_p)]


_lib = None


def load():
    """Load liblw.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"liblw is not built ({LIB_PATH} missing): run "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "lw_encode_bundle": ([P, P, P, P, P], i32),
        "lw_bundle_sections": ([P, P], i32),
        "lw_bundle_free": ([P], None),
        "lw_table_from_lengths": ([i32, P, i32, P, i32, P], i32),
        "lw_validate_sections": ([P, P], i32),
        "lw_workspace_bytes": ([P, i32], sz),
        "lw_decode": ([P, P, P, P], i32),
        "lw_decode_gemv": ([P, P, P, P, sz, P, P], i32),
        "lw_decode_gemm": ([P, P, i32, P, P, sz, P, P], i32),
        "lw_twin_gemv": ([P, P, P, P, sz, P, P], i32),
        "lw_twin_gemm": ([P, P, i32, P, P, sz, P, P], i32),
        "lw_status_string": ([i32], ctypes.c_char_p),
        "lw_last_error": ([], ctypes.c_char_p),
        "lw_version": ([], i32),
        "lw_decode_gemv_noalloc": ([P, P, P, P, P], i32),
        "lw_decode_gemv_group": ([P, i32, P, P, P, sz, P, P], i32),
        "lw_twin_gemv_group": ([P, i32, P, P, P, sz, P, P], i32),
        "lw_decode_gemm_group": ([P, i32, P, i32, P, P, sz, P, P], i32),
        "lw_twin_gemm_group": ([P, i32, P, i32, P, P, sz, P, P], i32),
        "lw_workspace_bytes_group": ([P, i32], sz),
        "lw_noalloc_scratch_bytes": ([], sz),
        "lw_bundle_desc": ([P, P], i32),
        "lw_bundle_serialized_bytes": ([P], sz),
        "lw_bundle_serialize": ([P, P, sz], i32),
        "lw_bundle_deserialize": ([P, sz, P], i32),
        "lw_bundle_save": ([P, ctypes.c_char_p], i32),
        "lw_bundle_load": ([ctypes.c_char_p, P], i32),
        "lw_transcode_twin": ([P, P, P, P], i32),
        "lw_decode_gemm_strips": ([P, P, i32, P, i32, P, P, sz, P, P], i32),
        "lw_twin_tile_rows": ([i32], i32),
        "lw_graph_begin": ([P], i32),
        "lw_graph_end": ([P, P], i32),
        "lw_graph_launch": ([P, P], i32),
        "lw_graph_free": ([P], None),
        "lw_table_lut_entries": ([P], i32),
        "lw_test_stall_next": ([i32], i32),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def _last_error() -> str:
    try:
        return load().lw_last_error().decode()
    except Exception:  # noqa: BLE001
        return ""


def _check(st: int, what: str):
    if st != 0:
        raise LwError(st, what)


def _np_ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------------------
# host bundles
# ----------------------------------------------------------------------------

@dataclass
class BundleStats:
    coded_bytes: int
    n_tiles: int
    n_verbatim: int
    max_tile_rows: int
    max_len: int
    min_len: int
    palette_size: int
    bits_per_weight: float
    lut_entries: int = 0


class HostBundle:
    """Owns an lw_bundle*; `sections` are numpy copies of its sections."""

    def __init__(self, handle, desc: LwDesc):
        self._h = handle
        self.desc = desc
        s = LwSections()
        _check(load().lw_bundle_sections(self._h, ctypes.byref(s)), "lw_bundle_sections")
        self.stats = BundleStats(int(s.coded_bytes), int(s.n_tiles), int(s.n_verbatim),
                                 int(s.max_tile_rows), int(s.max_len), int(s.min_len),
                                 int(s.palette_size), float(s.bits_per_weight),
                                 int(s.lut_entries))
        self.sections = {}
        for i, name in enumerate(SECTION_NAMES):
            n = int(s.bytes[i])
            if n:
                buf = (ctypes.c_uint8 * n).from_address(s.ptr[i])
                self.sections[name] = np.frombuffer(buf, dtype=np.uint8).copy()
        self._raw = s

    @property
    def fmt(self):
        return self.desc.fmt

    @property
    def twin(self):
        return bool(self.desc.twin)

    def view(self, name, dtype):
        return self.sections[name].view(dtype)

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.lw_bundle_free(self._h)
            self._h = None


def lw_encode_bundle(fmt: int, payload: np.ndarray, scales=None, mins=None,
                     twin: bool = False) -> HostBundle:
    """payload: uint8 codes [N][K] or uint16 bf16 bits [N][K]."""
    payload = np.ascontiguousarray(payload)
    n, k = payload.shape
    desc = LwDesc(fmt, int(twin), n, k)
    sc = None if scales is None else np.ascontiguousarray(scales, dtype=np.uint16)
    mn = None if mins is None else np.ascontiguousarray(mins, dtype=np.uint16)
    h = ctypes.c_void_p()
    _check(load().lw_encode_bundle(ctypes.byref(desc), _np_ptr(payload), _np_ptr(sc),
                                   _np_ptr(mn), ctypes.byref(h)), "lw_encode_bundle")
    return HostBundle(h, desc)


def _adopt(h) -> HostBundle:
    """Wrap a bundle handle returned by the library."""
    desc = LwDesc()
    st = load().lw_bundle_desc(h, ctypes.byref(desc))
    if st != 0:
        load().lw_bundle_free(h)
        raise LwError(st, "lw_bundle_desc")
    return HostBundle(h, desc)


def lw_bundle_serialize(hb: HostBundle) -> bytes:
    """The bundle as one byte string (the bundle file format)."""
    n = int(load().lw_bundle_serialized_bytes(hb._h))
    buf = ctypes.create_string_buffer(n)
    _check(load().lw_bundle_serialize(hb._h, buf, n), "lw_bundle_serialize")
    return buf.raw


def lw_bundle_deserialize(data: bytes) -> HostBundle:
    h = ctypes.c_void_p()
    _check(load().lw_bundle_deserialize(data, len(data), ctypes.byref(h)), "lw_bundle_deserialize")
    return _adopt(h)


def lw_bundle_save(hb: HostBundle, path) -> None:
    _check(load().lw_bundle_save(hb._h, os.fsencode(path)), "lw_bundle_save")


def lw_bundle_load(path) -> HostBundle:
    h = ctypes.c_void_p()
    _check(load().lw_bundle_load(os.fsencode(path), ctypes.byref(h)), "lw_bundle_load")
    return _adopt(h)


def lw_table_from_lengths(fmt: int, code_len, palette=None) -> np.ndarray:
    cl = np.ascontiguousarray(code_len, dtype=np.uint8)
    pal = None if palette is None else np.ascontiguousarray(palette, dtype=np.uint8)
    out = np.zeros(TABLE_BYTES, dtype=np.uint8)
    _check(load().lw_table_from_lengths(fmt, _np_ptr(cl), len(cl), _np_ptr(pal),
                                        0 if pal is None else len(pal), _np_ptr(out)),
           "lw_table_from_lengths")
    return out


def lw_table_lut_entries(table: np.ndarray) -> int:
    """Entries of the compact decode table the table-driven kernel builds from
    this lw_table (the lut_entries hint of a device bundle)."""
    t = np.ascontiguousarray(table, dtype=np.uint8)
    if t.size != TABLE_BYTES:
        raise LwError(1, "lw_table_lut_entries", f"a table is {TABLE_BYTES} bytes, got {t.size}")
    return int(load().lw_table_lut_entries(_np_ptr(t)))


def lw_test_stall_next(wait_us: int) -> None:
    """Testing hook: the next table-driven product launch leaves one stage
    unfilled and limits its waits to `wait_us` microseconds (it reports
    LW_DEV_TIMEOUT and finishes)."""
    _check(load().lw_test_stall_next(int(wait_us)), "lw_test_stall_next")


def table_fields(table: np.ndarray) -> dict:
    """Decode the documented lw_table layout (for tests and reports)."""
    t = np.asarray(table, dtype=np.uint8)
    i32 = t[:32].view(np.int32)
    return dict(fmt=int(i32[0]), alpha=int(i32[1]), n_sym=int(i32[2]), lmin=int(i32[3]),
                lmax=int(i32[4]), n_palette=int(i32[5]), phantom=int(i32[6]),
                lim_m1=t[32:80].view(np.uint32).copy(), off=t[80:128].view(np.int32).copy(),
                sym=t[128:640].view(np.uint16).copy(), code_len=t[640:896].copy(),
                palette=t[896:912].copy())


def lw_validate_sections(fmt: int, rows: int, cols: int, sections: dict, max_tile_rows: int,
                         twin: bool = False) -> None:
    desc = LwDesc(fmt, int(twin), rows, cols)
    s = LwSections()
    keep = []
    for i, name in enumerate(SECTION_NAMES):
        a = sections.get(name)
        if a is not None and a.size:
            a = np.ascontiguousarray(a).view(np.uint8)
            keep.append(a)
            s.ptr[i] = a.ctypes.data
            s.bytes[i] = a.nbytes
    s.max_tile_rows = max_tile_rows
    _check(load().lw_validate_sections(ctypes.byref(desc), ctypes.byref(s)),
           "lw_validate_sections")


# ----------------------------------------------------------------------------
# device bundles (caller-owned device memory: torch tensors)
# ----------------------------------------------------------------------------

class DeviceBundle:
    """Byte-for-byte device copies of a bundle's sections plus the
    lw_dev_bundle view that the C calls take."""

    def __init__(self, fmt, twin, rows, cols, sections: dict, max_tile_rows, lmin, lmax,
                 device="cuda", coded_bytes=None, lut_entries=None):
        """lut_entries: the compact decode table's size (lw_sections); None
        computes it from the host table section (lw_table_lut_entries)."""
        import torch
        if lut_entries is None:
            tab = sections.get("table")
            lut_entries = (lw_table_lut_entries(np.ascontiguousarray(tab).view(np.uint8).reshape(-1))
                           if tab is not None and not twin else 0)
        self.fmt, self.twin, self.rows, self.cols = fmt, bool(twin), rows, cols
        self.tensors = {}
        for name in SECTION_NAMES:
            a = sections.get(name)
            if a is not None and a.size:
                host = torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).copy())
                self.tensors[name] = host.to(device)
        self.coded_bytes = int(coded_bytes if coded_bytes is not None else
                               sum(t.numel() for t in self.tensors.values()))
        v = LwDevBundle()
        v.fmt, v.twin, v.rows, v.cols = fmt, int(twin), rows, cols
        v.max_tile_rows, v.lmin, v.lmax, v.lut_entries = max_tile_rows, lmin, lmax, lut_entries
        for name in SECTION_NAMES:
            t = self.tensors.get(name)
            setattr(v, name, t.data_ptr() if t is not None else None)
        self.view = v

    @classmethod
    def from_tensors(cls, fmt, twin, rows, cols, tensors: dict, max_tile_rows, lmin, lmax,
                     lut_entries=0):
        """A view over device tensors that already hold the sections."""
        self = cls.__new__(cls)
        self.fmt, self.twin, self.rows, self.cols = fmt, bool(twin), rows, cols
        self.tensors = dict(tensors)
        self.coded_bytes = int(sum(t.numel() * t.element_size() for t in self.tensors.values()))
        v = LwDevBundle()
        v.fmt, v.twin, v.rows, v.cols = fmt, int(twin), rows, cols
        v.max_tile_rows, v.lmin, v.lmax, v.lut_entries = max_tile_rows, lmin, lmax, lut_entries
        for name in SECTION_NAMES:
            t = self.tensors.get(name)
            setattr(v, name, t.data_ptr() if t is not None else None)
        self.view = v
        return self

    @classmethod
    def upload(cls, hb: HostBundle, device="cuda"):
        return cls(hb.desc.fmt, hb.desc.twin, hb.desc.rows, hb.desc.cols, hb.sections,
                   hb.stats.max_tile_rows, hb.stats.min_len, hb.stats.max_len, device,
                   hb.stats.coded_bytes, hb.stats.lut_entries)

    @property
    def ref(self):
        return ctypes.byref(self.view)


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _tp(t):
    """A tensor's address, unchecked (for callers that drive the C functions
    directly and check their buffers themselves)."""
    return ctypes.c_void_p(t.data_ptr())


# ----------------------------------------------------------------------------
# device buffers, checked before their addresses cross the C ABI
# ----------------------------------------------------------------------------
# The C calls take bare device addresses: they cannot tell how large a buffer
# is, whether it lives on the device or how it is strided.  A tensor that is
# too small, on the host or strided would let a kernel read or write outside
# it, so every tensor is checked here first (LW_ERR_INVALID_ARG, nothing
# launched).  Sizes follow the view's shape; a shape the library refuses
# anyway (not a multiple of 64 x 256) is left for it to report.

def _refuse(fn: str, detail: str):
    raise LwError(LW_ERR_INVALID_ARG, fn, detail)


def _buf(fn: str, name: str, t, nbytes: int, dtypes=None):
    """Address of tensor `t` after checking that it is a torch.Tensor of one
    of `dtypes` (any if None), contiguous and at least `nbytes` bytes.  Its
    device is checked afterwards (_on), once every buffer has passed."""
    import torch
    if not isinstance(t, torch.Tensor):
        _refuse(fn, f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if dtypes is not None and t.dtype not in dtypes:
        want = ", ".join(str(d).replace("torch.", "") for d in dtypes)
        _refuse(fn, f"{name}: dtype {str(t.dtype).replace('torch.', '')}, expected {want}")
    if not t.is_contiguous():
        _refuse(fn, f"{name}: not contiguous")
    have = t.numel() * t.element_size()
    if have < nbytes:
        _refuse(fn, f"{name}: {have} bytes, the call needs {nbytes}")
    return ctypes.c_void_p(t.data_ptr())


def _bundle_device(fn: str, db, name: str = "bundle"):
    """The one CUDA device holding every section tensor of `db`."""
    devs = {t.device for t in db.tensors.values()}
    if len(devs) != 1:
        _refuse(fn, f"{name}: sections on {sorted(map(str, devs)) or 'no device'}, "
                    "expected one CUDA device")
    dev = devs.pop()
    if dev.type != "cuda":
        _refuse(fn, f"{name}: sections on {dev}, expected a CUDA device")
    if not all(t.is_contiguous() for t in db.tensors.values()):
        _refuse(fn, f"{name}: a section tensor is not contiguous")
    return dev


def _on(fn: str, dev, *named):
    """Every (name, tensor) pair is on the bundle's device `dev`."""
    for name, t in named:
        if t.device.type != "cuda":
            _refuse(fn, f"{name}: on {t.device}, expected a CUDA device")
        if t.device != dev:
            _refuse(fn, f"{name}: on {t.device}, the bundle is on {dev}")


def _dims(db):
    """(N, K) of the view when the library accepts that shape, else (0, 0)."""
    n, k = int(db.view.rows), int(db.view.cols)
    return (n, k) if n > 0 and k > 0 and n % 64 == 0 and k % 256 == 0 else (0, 0)


def _act_types(fmt: int):
    """Activation dtypes and element size of a format (fp32; BF16 as
    bfloat16 or its bits)."""
    import torch
    if fmt == LW_FMT_BF16_EXP:
        return (torch.bfloat16, torch.int16) + ((torch.uint16,) if hasattr(torch, "uint16") else ()), 2
    if fmt in (LW_FMT_Q4_PAIR, LW_FMT_Q6):
        return (torch.float32,), 4
    return None, 0


def _decoded_bytes(fmt: int, n: int, k: int) -> int:
    """Bytes lw_decode writes: packed pairs (4-bit), one byte per code
    (6-bit), BF16 bits."""
    return {LW_FMT_Q4_PAIR: n * k // 2, LW_FMT_Q6: n * k, LW_FMT_BF16_EXP: 2 * n * k}.get(fmt, 0)


def _status_ptr(fn: str, d_status):
    import torch
    return _buf(fn, "d_status", d_status, 4, (torch.int32,))


def _ws_ptr(fn: str, ws):
    return _buf(fn, "ws", ws, 0), ctypes.c_size_t(ws.numel() * ws.element_size())


def _product_bufs(fn: str, db, x, y, batch: int, xname="x", yname="y"):
    """Checked addresses of one matrix's activations [batch][K] and outputs
    fp32 [batch][N] (devices not yet checked)."""
    import torch
    n, k = _dims(db)
    b = max(int(batch), 0)
    types, esize = _act_types(int(db.view.fmt))
    return (_buf(fn, xname, x, b * k * esize, types),
            _buf(fn, yname, y, b * n * 4, (torch.float32,)))


def _checked(fn: str, dbs, xs, ys, batch: int, ws, d_status, names=("x", "y"), indexed=False,
             extra=()):
    """Check a product call's buffers in two passes -- first every buffer's
    type, dtype, layout and size, then that the bundles and every buffer sit
    on one CUDA device -- and return the addresses: (x list, y list, ws,
    ws bytes, d_status).  `extra`: further (name, tensor) pairs whose device
    is checked."""
    n = len(dbs)
    if n < 1 or len(xs) != n or len(ys) != n:
        _refuse(fn, f"{n} bundles, {len(xs)} activations, {len(ys)} outputs")
    label = (lambda i: (f"{names[0]}[{i}]", f"{names[1]}[{i}]")) if indexed else (lambda i: names)
    bufs = [_product_bufs(fn, d, x, y, batch, *label(i)) for i, (d, x, y) in enumerate(zip(dbs, xs, ys))]
    wp, wb = _ws_ptr(fn, ws) if ws is not None else (None, None)
    sp = _status_ptr(fn, d_status)
    dev = _bundle_device(fn, dbs[0], "bundle[0]" if indexed else "bundle")
    for i in range(1, n):
        if _bundle_device(fn, dbs[i], f"bundle[{i}]") != dev:
            _refuse(fn, f"bundle[{i}]: not on {dev} like bundle[0]")
    named = [p for i in range(n) for p in zip(label(i), (xs[i], ys[i]))]
    _on(fn, dev, *named, *((("ws", ws),) if ws is not None else ()), ("d_status", d_status), *extra)
    return [b[0] for b in bufs], [b[1] for b in bufs], wp, wb, sp


def lw_workspace_bytes(db: DeviceBundle, batch: int = 1) -> int:
    return int(load().lw_workspace_bytes(db.ref, batch))


def lw_decode(db: DeviceBundle, out, d_status, stream=None) -> None:
    fn = "lw_decode"
    n, k = _dims(db)
    o = _buf(fn, "out", out, _decoded_bytes(int(db.view.fmt), n, k))
    sp = _status_ptr(fn, d_status)
    _on(fn, _bundle_device(fn, db), ("out", out), ("d_status", d_status))
    _check(load().lw_decode(db.ref, o, sp, _stream_ptr(stream)), fn)


def lw_decode_gemm_strips(db: DeviceBundle, strips, X, batch, Y, ws, d_status, stream=None) -> None:
    """Y = W X on the 64-row strips listed in `strips` (device int32 tensor,
    ascending); the other rows of Y are left as they are."""
    import torch
    fn = "lw_decode_gemm_strips"
    n = int(strips.numel()) if strips is not None else 0
    lp = _buf(fn, "strips", strips, 4 * n, (torch.int32,)) if n else None
    (xp,), (yp,), wp, wb, sp = _checked(fn, [db], [X], [Y], batch, ws, d_status, ("X", "Y"),
                                        extra=(("strips", strips),) if n else ())
    _check(load().lw_decode_gemm_strips(db.ref, lp, n, xp, batch, yp, wp, wb, sp,
                                        _stream_ptr(stream)), fn)


class PreparedGemv:
    """lw_decode_gemv (one matrix) or lw_decode_gemv_group (several) -- or
    their twins -- with the arguments marshalled once, for calls repeated
    every step: each call() is one C call.  The tensors must stay alive and
    in place."""

    def __init__(self, dbs, xs, ys, ws, d_status, twin: bool = False):
        lib = load()
        fn = "PreparedGemv"
        self._keep = (list(dbs), list(xs), list(ys), ws, d_status)
        n = len(dbs)
        xps, yps, self._ws, self._wsb, self._st = _checked(fn, dbs, xs, ys, 1, ws, d_status,
                                                           indexed=True)
        if n == 1:
            self._fn = lib.lw_twin_gemv if twin else lib.lw_decode_gemv
            self._args = (dbs[0].ref, xps[0], yps[0])
        else:
            self._fn = lib.lw_twin_gemv_group if twin else lib.lw_decode_gemv_group
            self._views = _views(dbs)
            self._xa = (ctypes.c_void_p * n)(*xps)
            self._ya = (ctypes.c_void_p * n)(*yps)
            self._args = (self._views, n, self._xa, self._ya)

    def __call__(self, stream=None) -> None:
        _check(self._fn(*self._args, self._ws, self._wsb, self._st, _stream_ptr(stream)),
               "prepared gemv")


class StepGraph:
    """Library calls captured once on a stream and replayed as one CUDA
    graph (lw_graph_begin / lw_graph_end / lw_graph_launch).  Use as
        g = StepGraph(stream)
        with g.capture():
            ...library calls on `stream` (e.g. with torch.cuda.stream(stream))...
        g.launch()"""

    def __init__(self, stream):
        self.stream = stream
        self._h = ctypes.c_void_p()

    def capture(self):
        import contextlib
        import torch

        @contextlib.contextmanager
        def cm():
            with torch.cuda.stream(self.stream):
                _check(load().lw_graph_begin(_stream_ptr(self.stream)), "lw_graph_begin")
                try:
                    yield self
                finally:
                    _check(load().lw_graph_end(_stream_ptr(self.stream), ctypes.byref(self._h)),
                           "lw_graph_end")
        return cm()

    def launch(self, stream=None) -> None:
        _check(load().lw_graph_launch(self._h, _stream_ptr(stream if stream is not None else self.stream)),
               "lw_graph_launch")

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value and _lib is not None:
            _lib.lw_graph_free(self._h)
            self._h = ctypes.c_void_p()


def lw_twin_tile_rows(fmt: int) -> int:
    return int(load().lw_twin_tile_rows(fmt))


def lw_transcode_twin(db: DeviceBundle, d_status, stream=None) -> DeviceBundle:
    """Transcode a coded device bundle into its fixed-width twin on the
    device: new words, tile offsets and lane bit counts; every other section
    is the coded bundle's own tensor (shared, not copied)."""
    import torch
    dev = db.tensors["tile_off"].device
    n_tiles = (db.rows // 64) * (db.cols // 256)
    r2 = lw_twin_tile_rows(db.fmt)
    t = {"words": torch.empty(n_tiles * r2 * 128, dtype=torch.uint8, device=dev),
         "tile_off": torch.empty((n_tiles + 1) * 4, dtype=torch.uint8, device=dev),
         "lane_bits": torch.empty(n_tiles * 64, dtype=torch.uint8, device=dev)}
    for name in ("table", "qparams", "signman", "vflags", "vrow_off", "vexp"):
        if name in db.tensors:
            t[name] = db.tensors[name]
    tw = DeviceBundle.from_tensors(db.fmt, True, db.rows, db.cols, t, r2, 0, 0)
    fn = "lw_transcode_twin"
    sp = _status_ptr(fn, d_status)
    _on(fn, _bundle_device(fn, db), ("d_status", d_status))
    _check(load().lw_transcode_twin(db.ref, tw.ref, sp, _stream_ptr(stream)), fn)
    return tw


def _gemv(fn, db, x, y, ws, d_status, stream):
    (xp,), (yp,), wp, wb, sp = _checked(fn, [db], [x], [y], 1, ws, d_status)
    _check(getattr(load(), fn)(db.ref, xp, yp, wp, wb, sp, _stream_ptr(stream)), fn)


def _gemm(fn, db, X, batch, Y, ws, d_status, stream):
    (xp,), (yp,), wp, wb, sp = _checked(fn, [db], [X], [Y], batch, ws, d_status, ("X", "Y"))
    _check(getattr(load(), fn)(db.ref, xp, batch, yp, wp, wb, sp, _stream_ptr(stream)), fn)


def lw_decode_gemv(db: DeviceBundle, x, y, ws, d_status, stream=None) -> None:
    _gemv("lw_decode_gemv", db, x, y, ws, d_status, stream)


def lw_decode_gemm(db: DeviceBundle, X, batch, Y, ws, d_status, stream=None) -> None:
    _gemm("lw_decode_gemm", db, X, batch, Y, ws, d_status, stream)


def lw_twin_gemv(db: DeviceBundle, x, y, ws, d_status, stream=None) -> None:
    _gemv("lw_twin_gemv", db, x, y, ws, d_status, stream)


def lw_twin_gemm(db: DeviceBundle, X, batch, Y, ws, d_status, stream=None) -> None:
    _gemm("lw_twin_gemm", db, X, batch, Y, ws, d_status, stream)


def lw_decode_gemv_noalloc(db: DeviceBundle, x, y, d_status, stream=None) -> None:
    """lw_decode_gemv with the library's fixed device scratch instead of a
    caller workspace (allocates nothing)."""
    fn = "lw_decode_gemv_noalloc"
    (xp,), (yp,), _, _, sp = _checked(fn, [db], [x], [y], 1, None, d_status)
    _check(load().lw_decode_gemv_noalloc(db.ref, xp, yp, sp, _stream_ptr(stream)), fn)


def _views(dbs):
    arr = (ctypes.c_void_p * len(dbs))(*[ctypes.addressof(d.view) for d in dbs])
    return arr


def lw_workspace_bytes_group(dbs) -> int:
    return int(load().lw_workspace_bytes_group(_views(dbs), len(dbs)))


def _gemv_group(fn, dbs, xs, ys, ws, d_status, stream):
    xps, yps, wp, wb, sp = _checked(fn, dbs, xs, ys, 1, ws, d_status, indexed=True)
    n = len(dbs)
    xa, ya = (ctypes.c_void_p * n)(*xps), (ctypes.c_void_p * n)(*yps)
    _check(getattr(load(), fn)(_views(dbs), n, xa, ya, wp, wb, sp, _stream_ptr(stream)), fn)


def _gemm_group(fn, dbs, Xs, batch, Ys, ws, d_status, stream):
    xps, yps, wp, wb, sp = _checked(fn, dbs, Xs, Ys, batch, ws, d_status, indexed=True)
    n = len(dbs)
    xa, ya = (ctypes.c_void_p * n)(*xps), (ctypes.c_void_p * n)(*yps)
    _check(getattr(load(), fn)(_views(dbs), n, xa, batch, ya, wp, wb, sp, _stream_ptr(stream)), fn)


def lw_decode_gemm_group(dbs, Xs, batch, Ys, ws, d_status, stream=None) -> None:
    """One launch for several 4-/6-bit matrices, batch 1..8: Ys[i] = Xs[i] W_i^T."""
    _gemm_group("lw_decode_gemm_group", dbs, Xs, batch, Ys, ws, d_status, stream)


def lw_twin_gemm_group(dbs, Xs, batch, Ys, ws, d_status, stream=None) -> None:
    _gemm_group("lw_twin_gemm_group", dbs, Xs, batch, Ys, ws, d_status, stream)


def lw_decode_gemv_group(dbs, xs, ys, ws, d_status, stream=None) -> None:
    """One launch for several 4-/6-bit matrices: ys[i] = W_i xs[i]."""
    _gemv_group("lw_decode_gemv_group", dbs, xs, ys, ws, d_status, stream)


def lw_twin_gemv_group(dbs, xs, ys, ws, d_status, stream=None) -> None:
    """The fixed-width twin of lw_decode_gemv_group."""
    _gemv_group("lw_twin_gemv_group", dbs, xs, ys, ws, d_status, stream)


def lw_noalloc_scratch_bytes() -> int:
    return int(load().lw_noalloc_scratch_bytes())
