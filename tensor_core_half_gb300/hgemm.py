"""Python binding of the C ABI in include/hgemm.h (ctypes; marshalling only).

Every function here converts Python arguments to the C types and calls the
entry point of the same name in libhgemm.so; all computation runs in the CUDA
kernels behind it.  Importing this module fails loudly when the library has
not been built: there is no fallback.

``matmul`` is a convenience for torch tensors: it reads shapes, dtypes, device
pointers and the current stream, allocates C with torch and calls hgemm_run.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhgemm.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "hgemm.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        "libhgemm.so is not built (expected at %s). Build it with `python -m tensor_core_half_gb300.build` "
        "or `python -c 'import __graft_entry__ as g; g.build()'`." % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

# ---------------------------------------------------------------- enums ----
HGEMM_OK = 0
HGEMM_ERR_INVALID_ARG = 1
HGEMM_ERR_UNSUPPORTED = 2
HGEMM_ERR_MISALIGNED = 3
HGEMM_ERR_ALIAS = 4
HGEMM_ERR_NO_DEVICE = 5
HGEMM_ERR_CUDA = 6
HGEMM_ERR_TIMEOUT = 7
HGEMM_ERR_OOM = 8

HGEMM_LAYOUT_TN = 0
HGEMM_LAYOUT_NN = 1

HGEMM_F16 = 0
HGEMM_BF16 = 1
HGEMM_F32 = 2

HGEMM_VARIANT_AUTO = 0
HGEMM_VARIANT_1SM_128x128 = 1
HGEMM_VARIANT_1SM_128x256 = 2
HGEMM_VARIANT_2SM_256x256 = 3
HGEMM_VARIANT_SPLITK = 4
HGEMM_VARIANT_2SM_256x192 = 5

HGEMM_OPT_FORCE_VARIANT = 1
HGEMM_OPT_TIMEOUT_NS = 2
HGEMM_OPT_INJECT_FAULT = 3
HGEMM_OPT_GROUP_M = 4
HGEMM_OPT_MAX_CTAS = 5
HGEMM_OPT_STREAM_K = 6
HGEMM_OPT_TRACE = 7
HGEMM_OPT_SCHEDULE = 8
HGEMM_SCHEDULE_STATIC = 0
HGEMM_SCHEDULE_DYNAMIC = 1
SCHEDULES = {"static": HGEMM_SCHEDULE_STATIC, "dynamic": HGEMM_SCHEDULE_DYNAMIC}
HGEMM_OPT_EPILOGUE = 9
HGEMM_EPILOGUE_TMA_STORE = 0
HGEMM_EPILOGUE_DIRECT = 1
EPILOGUES = {"tma": HGEMM_EPILOGUE_TMA_STORE, "direct": HGEMM_EPILOGUE_DIRECT}
HGEMM_OPT_CHECKS = 10
HGEMM_OPT_TRACE_ITEMS = 11
HGEMM_ERR_CHECK = 9
HGEMM_CHECK_WORK_ID, HGEMM_CHECK_ITEM, HGEMM_CHECK_TICKET, HGEMM_CHECK_CONTRIBUTOR, HGEMM_CHECK_PARTIAL = 1, 2, 3, 4, 5

LAYOUTS = {"TN": HGEMM_LAYOUT_TN, "NN": HGEMM_LAYOUT_NN}
DTYPES = {"f16": HGEMM_F16, "bf16": HGEMM_BF16, "f32": HGEMM_F32}
VARIANTS = {"auto": HGEMM_VARIANT_AUTO, "1sm128": HGEMM_VARIANT_1SM_128x128, "1sm256": HGEMM_VARIANT_1SM_128x256,
            "2sm256": HGEMM_VARIANT_2SM_256x256, "splitk": HGEMM_VARIANT_SPLITK, "2sm192": HGEMM_VARIANT_2SM_256x192}


class hgemm_plan_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "variant", "cta_group", "tile_m", "tile_n", "block_k", "stages", "tiles_m", "tiles_n", "num_tiles",
        "k_blocks", "grid", "group_m", "smem_bytes", "tmem_cols")] + [
        ("workspace_bytes", ctypes.c_int64), ("dp_tiles", ctypes.c_int32), ("stream_k", ctypes.c_int32),
        ("sk_units", ctypes.c_int64), ("sk_ranges", ctypes.c_int32), ("work_ids", ctypes.c_int32),
        ("schedule", ctypes.c_int32), ("splitk_chunks", ctypes.c_int32), ("splitk_head_units", ctypes.c_int64),
        ("splitk_align", ctypes.c_int32), ("sk_pieces", ctypes.c_int32)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_u32 = ctypes.c_uint32
_u64 = ctypes.c_uint64

_lib.hgemm_create.restype = _i32
_lib.hgemm_create.argtypes = [ctypes.POINTER(_vp)]
_lib.hgemm_destroy.restype = _i32
_lib.hgemm_destroy.argtypes = [_vp]
_lib.hgemm_run.restype = _i32
_lib.hgemm_run.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _i32, _i32, _vp]
_lib.hgemm_run_host.restype = _i32
_lib.hgemm_run_host.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _i32, _i32, _vp]
_lib.hgemm_sync_status.restype = _i32
_lib.hgemm_sync_status.argtypes = [_vp, _vp, ctypes.POINTER(_i32)]
_lib.hgemm_set_option.restype = _i32
_lib.hgemm_set_option.argtypes = [_vp, _i32, _i64]
_lib.hgemm_status_string.restype = ctypes.c_char_p
_lib.hgemm_status_string.argtypes = [_i32]
_lib.hgemm_plan_ex.restype = _i32
_lib.hgemm_plan_ex.argtypes = [_i64, _i64, _i64, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                               ctypes.POINTER(hgemm_plan_t)]
_lib.hgemm_plan.restype = _i32
_lib.hgemm_plan.argtypes = [_i64, _i64, _i64, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                            ctypes.POINTER(hgemm_plan_t)]
_lib.hgemm_plan_work_item.restype = _i32
_lib.hgemm_plan_work_item.argtypes = [ctypes.POINTER(hgemm_plan_t), _i32, _i32] + [ctypes.POINTER(_i32)] * 4
_lib.hgemm_plan_id_item.restype = _i32
_lib.hgemm_plan_id_item.argtypes = [ctypes.POINTER(hgemm_plan_t), _i32, _i32] + [ctypes.POINTER(_i32)] * 4
_lib.hgemm_tma_bench.restype = _i32
_lib.hgemm_tma_bench.argtypes = [_vp, _i64, _i64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                 _vp]
_lib.hgemm_plan_tile.restype = _i32
_lib.hgemm_plan_tile.argtypes = [ctypes.POINTER(hgemm_plan_t), _i32, ctypes.POINTER(_i32), ctypes.POINTER(_i32)]
_lib.hgemm_plan_splitk_range.restype = _i32
_lib.hgemm_plan_splitk_range.argtypes = [ctypes.POINTER(hgemm_plan_t), _i32, ctypes.POINTER(_i64),
                                         ctypes.POINTER(_i64)]
_lib.hgemm_plan_splitk_segment.restype = _i32
_lib.hgemm_plan_splitk_segment.argtypes = [ctypes.POINTER(hgemm_plan_t), _i32, _i32] + [ctypes.POINTER(_i32)] * 4
_lib.hgemm_encode_idesc.restype = _u32
_lib.hgemm_encode_idesc.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32]
_lib.hgemm_encode_smem_desc.restype = _u64
_lib.hgemm_encode_smem_desc.argtypes = [_u32, _u32, _u32, _i32]
_lib.hgemm_version.restype = _i32
_lib.hgemm_version.argtypes = []
_lib.hgemm_run_splitk_noalloc.restype = _i32
_lib.hgemm_run_splitk_noalloc.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _vp]


class hgemm_trace_record_t(ctypes.Structure):
    _fields_ = [("t_ns", ctypes.c_uint64), ("cta", ctypes.c_uint32), ("role", ctypes.c_uint16),
                ("kind", ctypes.c_uint16), ("item", ctypes.c_int32), ("value", ctypes.c_int32)]


_lib.hgemm_trace_read.restype = _i32
_lib.hgemm_trace_read.argtypes = [_vp, ctypes.POINTER(hgemm_trace_record_t), _i64, ctypes.POINTER(_i64)]


class HgemmError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = int(status)
        super().__init__("%s%s" % (where + ": " if where else "", hgemm_status_string(status)))


def lib():
    """The loaded ctypes library (for symbol checks)."""
    return _lib


def declared_functions():
    """Names of the functions declared in include/hgemm.h."""
    with open(HEADER_PATH) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(hgemm_[a-z_0-9]+)\s*\(", text,
                                 flags=re.M)))


# ------------------------------------------------------- entry points ----
def hgemm_status_string(status) -> str:
    return _lib.hgemm_status_string(int(status)).decode()


def hgemm_version() -> int:
    return int(_lib.hgemm_version())


def hgemm_create() -> int:
    h = _vp()
    st = _lib.hgemm_create(ctypes.byref(h))
    if st != HGEMM_OK:
        raise HgemmError(st, "hgemm_create")
    return h.value


def hgemm_destroy(h) -> int:
    return int(_lib.hgemm_destroy(h))


def hgemm_run(h, A, B, C, M, N, K, layout, in_dtype, acc_dtype, out_dtype, stream=0) -> int:
    return int(_lib.hgemm_run(h, A, B, C, int(M), int(N), int(K), int(layout), int(in_dtype), int(acc_dtype),
                              int(out_dtype), stream))


def hgemm_run_host(h, A, B, C, M, N, K, layout, in_dtype, acc_dtype, out_dtype, stream=0) -> int:
    """End-to-end product on host buffers (see include/hgemm.h)."""
    return int(_lib.hgemm_run_host(h, A, B, C, int(M), int(N), int(K), int(layout), int(in_dtype), int(acc_dtype),
                                   int(out_dtype), stream))


def hgemm_sync_status(h, stream=0):
    d = _i32(0)
    st = _lib.hgemm_sync_status(h, stream, ctypes.byref(d))
    return int(st), int(d.value)


def hgemm_set_option(h, option, value) -> int:
    return int(_lib.hgemm_set_option(h, int(option), int(value)))


def hgemm_plan(M, N, K, layout=HGEMM_LAYOUT_TN, in_dtype=HGEMM_BF16, acc_dtype=HGEMM_F32, out_dtype=HGEMM_BF16,
               num_sms=152, variant=HGEMM_VARIANT_AUTO, group_m=0, stream_k=1, schedule=None):
    """hgemm_plan, or hgemm_plan_ex when a schedule is given."""
    p = hgemm_plan_t()
    if schedule is None:
        st = _lib.hgemm_plan(int(M), int(N), int(K), int(layout), int(in_dtype), int(acc_dtype), int(out_dtype),
                             int(num_sms), int(variant), int(group_m), int(stream_k), ctypes.byref(p))
    else:
        st = _lib.hgemm_plan_ex(int(M), int(N), int(K), int(layout), int(in_dtype), int(acc_dtype), int(out_dtype),
                                int(num_sms), int(variant), int(group_m), int(stream_k), int(schedule),
                                ctypes.byref(p))
    return int(st), p


def hgemm_plan_work_item(plan, cluster, index):
    t, a, b, s = _i32(), _i32(), _i32(), _i32()
    st = _lib.hgemm_plan_work_item(ctypes.byref(plan), int(cluster), int(index), ctypes.byref(t), ctypes.byref(a),
                                   ctypes.byref(b), ctypes.byref(s))
    return int(st), t.value, a.value, b.value, s.value


def hgemm_plan_id_item(plan, id, index):
    t, a, b, s = _i32(), _i32(), _i32(), _i32()
    st = _lib.hgemm_plan_id_item(ctypes.byref(plan), int(id), int(index), ctypes.byref(t), ctypes.byref(a),
                                 ctypes.byref(b), ctypes.byref(s))
    return int(st), t.value, a.value, b.value, s.value


HGEMM_TMA_2D_16B, HGEMM_TMA_3D_16B, HGEMM_TMA_2D_128B, HGEMM_TMA_3D_128B, HGEMM_TMA_BULK = range(5)
TMA_MODES = {"2d_16b": HGEMM_TMA_2D_16B, "3d_16b": HGEMM_TMA_3D_16B, "2d_128b": HGEMM_TMA_2D_128B,
             "3d_128b": HGEMM_TMA_3D_128B, "bulk": HGEMM_TMA_BULK}


class hgemm_tma_bench_config_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("mode", "tile_rows", "tile_cols", "depth", "issuers", "ctas", "iters",
                                              "walk")]


class hgemm_tma_bench_result_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in ("ms", "bytes", "gbs", "bytes_per_clk_sm", "sm_mhz")] + [
        (n, ctypes.c_int32) for n in ("copies_per_tile", "ctas", "tile_bytes", "reserved")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_ if n != "reserved"}


HGEMM_TMA_WALK_SCATTERED, HGEMM_TMA_WALK_ALONG_K = 0, 1
TMA_WALKS = {"scattered": HGEMM_TMA_WALK_SCATTERED, "along_k": HGEMM_TMA_WALK_ALONG_K}


def hgemm_tma_bench(src_ptr, height, width, mode, tile_rows, tile_cols, depth, iters, issuers=1, ctas=0, stream=0,
                    max_ctas=1024, walk=0):
    """Runs the TMA micro-benchmark (synchronous).  Returns (status, result,
    sums [ctas][2], last_tiles [ctas][depth]) with plain Python containers."""
    cfg = hgemm_tma_bench_config_t(int(mode), int(tile_rows), int(tile_cols), int(depth), int(issuers), int(ctas),
                                   int(iters), int(walk))
    res = hgemm_tma_bench_result_t()
    n = max_ctas if ctas == 0 else int(ctas)
    sums = (ctypes.c_uint64 * (2 * n))()
    last = (ctypes.c_int32 * (max(1, int(depth)) * n))()
    st = _lib.hgemm_tma_bench(src_ptr, int(height), int(width), ctypes.byref(cfg), ctypes.byref(res), sums, last,
                              stream)
    got = res.ctas if st == HGEMM_OK else 0
    return (int(st), res, [(sums[2 * i], sums[2 * i + 1]) for i in range(got)],
            [list(last[i * depth:(i + 1) * depth]) for i in range(got)])


def hgemm_plan_tile(plan, t):
    m, n = _i32(), _i32()
    st = _lib.hgemm_plan_tile(ctypes.byref(plan), int(t), ctypes.byref(m), ctypes.byref(n))
    return int(st), m.value, n.value


def hgemm_plan_splitk_range(plan, cta):
    b, e = _i64(), _i64()
    st = _lib.hgemm_plan_splitk_range(ctypes.byref(plan), int(cta), ctypes.byref(b), ctypes.byref(e))
    return int(st), b.value, e.value


def hgemm_plan_splitk_segment(plan, chunk, index):
    t, k0, k1, f = _i32(), _i32(), _i32(), _i32()
    st = _lib.hgemm_plan_splitk_segment(ctypes.byref(plan), int(chunk), int(index), ctypes.byref(t), ctypes.byref(k0),
                                        ctypes.byref(k1), ctypes.byref(f))
    return int(st), t.value, k0.value, k1.value, f.value


def hgemm_encode_idesc(mma_m, mma_n, in_dtype, acc_dtype, a_mn_major=0, b_mn_major=0) -> int:
    return int(_lib.hgemm_encode_idesc(int(mma_m), int(mma_n), int(in_dtype), int(acc_dtype), int(a_mn_major),
                                       int(b_mn_major)))


def hgemm_encode_smem_desc(addr, lbo, sbo, swizzle) -> int:
    return int(_lib.hgemm_encode_smem_desc(int(addr), int(lbo), int(sbo), int(swizzle)))


def hgemm_run_splitk_noalloc(A, B, C, M, N, K, in_dtype, out_dtype, stream=0) -> int:
    """Skinny-M product with scratch in a fixed device array: no allocation,
    no handle (for callers that cannot allocate device memory)."""
    return int(_lib.hgemm_run_splitk_noalloc(A, B, C, int(M), int(N), int(K), int(in_dtype), int(out_dtype), stream))


def hgemm_trace_read(h, capacity):
    """Returns (status, events recorded, list of (t_ns, cta, role, kind, item, value))."""
    buf = (hgemm_trace_record_t * max(1, int(capacity)))()
    n = _i64(0)
    st = _lib.hgemm_trace_read(h, buf, int(capacity), ctypes.byref(n))
    rows = [(r.t_ns, r.cta, r.role, r.kind, r.item, r.value) for r in buf[:min(int(capacity), n.value)]] \
        if st == HGEMM_OK else []
    return int(st), int(n.value), rows


# ------------------------------------------------------ torch helpers ----
_local = threading.local()


def _default_handle():
    h = getattr(_local, "handle", None)
    if h is None:
        h = Handle()
        _local.handle = h
    return h


class Handle:
    """Owns an hgemm handle bound to the current CUDA device."""

    def __init__(self):
        self.h = hgemm_create()

    def close(self):
        if self.h:
            hgemm_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def set_option(self, option, value):
        st = hgemm_set_option(self.h, option, value)
        if st != HGEMM_OK:
            raise HgemmError(st, "hgemm_set_option")

    def sync_status(self, stream=None):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream()
        return hgemm_sync_status(self.h, s.cuda_stream)

    def run(self, A, B, C, layout="TN", acc="f32", stream=None, check=True):
        """C = A . B on torch CUDA tensors (A [M,K]; B [N,K] for TN or [K,N] for NN; C [M,N])."""
        import torch
        M, N, K = operand_shape(A, B, C, layout, cuda=True)
        s = stream if stream is not None else torch.cuda.current_stream()
        st = hgemm_run(self.h, A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, LAYOUTS[layout],
                       _torch_dtype(A.dtype), DTYPES[acc], _torch_dtype(C.dtype), s.cuda_stream)
        if check and st != HGEMM_OK:
            raise HgemmError(st, "hgemm_run")
        return st


def operand_shape(A, B, C, layout, cuda):
    """(M, N, K) of C = A . B after checking that the three tensors describe one
    product the C ABI can take: 2-D, packed row-major (contiguous), on the right
    side (CUDA tensors for hgemm_run, host tensors for hgemm_run_host), A and B
    of one element type, B [N,K] (TN) or [K,N] (NN) with A's K, C [M,N].  The
    library receives bare pointers and sizes, so a view that breaks any of these
    would otherwise be read as something else; ValueError names the mismatch."""
    if layout not in LAYOUTS:
        raise ValueError("layout must be one of %s" % sorted(LAYOUTS))
    for name, t in (("A", A), ("B", B), ("C", C)):
        if t.dim() != 2:
            raise ValueError("%s must be 2-D, got shape %s" % (name, tuple(t.shape)))
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous (packed row-major)" % name)
        if bool(t.is_cuda) != cuda:
            raise ValueError("%s must be a %s tensor" % (name, "CUDA" if cuda else "host (CPU)"))
    if A.dtype != B.dtype:
        raise ValueError("A and B must share one element type, got %s and %s" % (A.dtype, B.dtype))
    M, K = A.shape
    N, Kb = (B.shape[0], B.shape[1]) if layout == "TN" else (B.shape[1], B.shape[0])
    if Kb != K:
        raise ValueError("B holds K = %d for layout %s, A holds K = %d" % (Kb, layout, K))
    if tuple(C.shape) != (M, N):
        raise ValueError("C must be [%d, %d], got %s" % (M, N, tuple(C.shape)))
    return int(M), int(N), int(K)


def _run_host_method(self, A, B, C, layout="TN", acc="f32", stream=None, check=True):
    """C = A . B on CPU tensors (pinned for overlap); returns once enqueued."""
    import torch
    M, N, K = operand_shape(A, B, C, layout, cuda=False)
    s = stream if stream is not None else torch.cuda.current_stream()
    st = hgemm_run_host(self.h, A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, LAYOUTS[layout],
                        _torch_dtype(A.dtype), DTYPES[acc], _torch_dtype(C.dtype), s.cuda_stream)
    if check and st != HGEMM_OK:
        raise HgemmError(st, "hgemm_run_host")
    return st


Handle.run_host = _run_host_method


def _torch_dtype(dt):
    import torch
    if dt == torch.float16:
        return HGEMM_F16
    if dt == torch.bfloat16:
        return HGEMM_BF16
    if dt == torch.float32:
        return HGEMM_F32
    raise TypeError("unsupported dtype %s" % dt)


def matmul(A, B, layout="TN", acc="f32", out_dtype=None, out=None, handle=None, stream=None):
    """Returns C = A . B (torch CUDA tensors, contiguous).  See Handle.run."""
    import torch
    if not (A.is_cuda and B.is_cuda):
        raise ValueError("matmul needs CUDA tensors; there is no CPU path")
    if not (A.is_contiguous() and B.is_contiguous()):
        raise ValueError("A and B must be contiguous")
    M = A.shape[0]
    N = B.shape[0] if layout == "TN" else B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or A.dtype, device=A.device)
    (handle or _default_handle()).run(A, B, out, layout=layout, acc=acc, stream=stream)
    return out
