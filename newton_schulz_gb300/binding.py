"""Thin ctypes binding of libmuon (include/muon.h): argument marshalling only.

Every step of the Muon path runs in the library's CUDA kernels; this module
only turns tensors into pointers, shapes and a stream handle.  Loading fails
loudly when the library has not been built (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os
from typing import Iterable, Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmuon.so")

MUON_OK = 0
STATUS_NAMES = {
    0: "MUON_OK", 1: "MUON_ERR_INVALID_ARGUMENT", 2: "MUON_ERR_UNSUPPORTED",
    3: "MUON_ERR_ALIAS", 4: "MUON_ERR_OUT_OF_MEMORY", 5: "MUON_ERR_CUDA",
    6: "MUON_ERR_TIMEOUT", 7: "MUON_ERR_NONFINITE", 8: "MUON_ERR_BOUNDS",
}
MUON_F32, MUON_BF16 = 0, 1
SCALE_SQRT_MAX1_R_OVER_C, SCALE_RMS_0P2_SQRT_MAXDIM, SCALE_ONE = 0, 1, 2
NS_BF16, NS_TF32 = 0, 1
PROFILE_KINDS = ("prep", "gram", "poly", "apply", "update", "fused_small", "adamw")

EXPORTED = (
    "muon_ns_default_config", "muon_ns_batched", "muon_ns_batched_ex", "muon_step_grouped",
    "muon_step_grouped_ex", "muon_step_grouped_host", "muon_query_status", "muon_status_string",
    "muon_release_workspace", "muon_last_launch_count", "muon_profile_enable",
    "muon_profile_read", "muon_adamw_grouped", "muon_ns_cost_table", "muon_assign_owners",
    "muon_ns_batched_noalloc", "muon_debug_inject_stall", "muon_debug_guard_check",
    "muon_ns_path",
    "muon_ns_gram_restart",
    "muon_debug_build",
)
PATH_SMALL, PATH_XSPACE, PATH_GRAM_SPACE = 0, 1, 2
INJECT_NONE, INJECT_GEMM, INJECT_SMALL = 0, 1, 2


class MuonError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")
        self.code = code


class NsConfig(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int32), ("coeffs", ctypes.POINTER(ctypes.c_float)),
                ("a", ctypes.c_float), ("b", ctypes.c_float), ("c", ctypes.c_float),
                ("eps", ctypes.c_float), ("precision", ctypes.c_int32)]


class Group(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("w_dtype", ctypes.c_int32),
                ("G", ctypes.c_void_p), ("g_dtype", ctypes.c_int32),
                ("Mom", ctypes.c_void_p),
                ("B", ctypes.c_int64), ("M", ctypes.c_int64), ("N", ctypes.c_int64)]


class AdamwGroup(ctypes.Structure):
    _fields_ = [("param", ctypes.c_void_p), ("p_dtype", ctypes.c_int32),
                ("grad", ctypes.c_void_p), ("g_dtype", ctypes.c_int32),
                ("exp_avg", ctypes.c_void_p), ("exp_avg_sq", ctypes.c_void_p),
                ("numel", ctypes.c_int64)]


class AdamwConfig(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("step", ctypes.c_int64)]


class Unit(ctypes.Structure):
    _fields_ = [("cost", ctypes.c_double), ("bytes", ctypes.c_int64), ("elems", ctypes.c_int64),
                ("layer", ctypes.c_int32)]


_lib = None


def load(path: str = None) -> ctypes.CDLL:
    """Load libmuon.so, or the library MUON_LIB_PATH names (the -DMUON_DEBUG
    build, libmuon_debug.so); raises OSError when it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("MUON_LIB_PATH") or LIB_PATH
    if not os.path.exists(path):
        raise OSError(f"{path} not found: build it with `python -m newton_schulz_gb300.build`")
    lib = ctypes.CDLL(path)
    i32, i64, vp, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
    lib.muon_ns_default_config.argtypes = [ctypes.POINTER(NsConfig)]
    lib.muon_ns_default_config.restype = i32
    lib.muon_ns_batched.argtypes = [vp, i64, i64, i64, ctypes.c_int, f32, f32, f32, vp]
    lib.muon_ns_batched.restype = i32
    lib.muon_ns_batched_ex.argtypes = [vp, i32, i64, i64, i64, ctypes.POINTER(NsConfig), vp, vp]
    lib.muon_ns_batched_ex.restype = i32
    lib.muon_step_grouped.argtypes = [ctypes.POINTER(Group), ctypes.c_int, f32, ctypes.c_int,
                                      f32, f32, ctypes.c_int, vp]
    lib.muon_step_grouped.restype = i32
    lib.muon_step_grouped_ex.argtypes = [ctypes.POINTER(Group), ctypes.c_int, f32, ctypes.c_int,
                                         f32, f32, ctypes.c_int, ctypes.POINTER(NsConfig), vp]
    lib.muon_step_grouped_ex.restype = i32
    lib.muon_adamw_grouped.argtypes = [ctypes.POINTER(AdamwGroup), ctypes.c_int,
                                       ctypes.POINTER(AdamwConfig), vp]
    lib.muon_adamw_grouped.restype = i32
    lib.muon_ns_cost_table.argtypes = [ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                                       ctypes.POINTER(NsConfig), ctypes.c_int,
                                       ctypes.POINTER(ctypes.c_double), vp]
    lib.muon_ns_cost_table.restype = i32
    lib.muon_assign_owners.argtypes = [ctypes.POINTER(Unit), ctypes.c_int, ctypes.c_int,
                                       ctypes.c_double, ctypes.POINTER(ctypes.c_int32)]
    lib.muon_assign_owners.restype = i32
    lib.muon_step_grouped_host.argtypes = lib.muon_step_grouped_ex.argtypes
    lib.muon_step_grouped_host.restype = i32
    lib.muon_ns_batched_noalloc.argtypes = [vp, i64, i64, i64, ctypes.c_int, f32, f32, f32, vp]
    lib.muon_ns_batched_noalloc.restype = i32
    lib.muon_debug_inject_stall.argtypes = [ctypes.c_int]
    lib.muon_debug_inject_stall.restype = i32
    lib.muon_ns_path.argtypes = [i64, i64, ctypes.POINTER(NsConfig)]
    lib.muon_ns_path.restype = ctypes.c_int
    lib.muon_ns_gram_restart.argtypes = [i64]
    lib.muon_ns_gram_restart.restype = ctypes.c_int
    lib.muon_debug_build.argtypes = []
    lib.muon_debug_build.restype = ctypes.c_int
    lib.muon_debug_guard_check.argtypes = [vp, ctypes.POINTER(ctypes.c_int64)]
    lib.muon_debug_guard_check.restype = i32
    lib.muon_query_status.argtypes = [vp]
    lib.muon_query_status.restype = i32
    lib.muon_status_string.argtypes = [i32]
    lib.muon_status_string.restype = ctypes.c_char_p
    lib.muon_release_workspace.argtypes = []
    lib.muon_release_workspace.restype = None
    lib.muon_last_launch_count.argtypes = []
    lib.muon_last_launch_count.restype = ctypes.c_int
    lib.muon_profile_enable.argtypes = [ctypes.c_int]
    lib.muon_profile_enable.restype = ctypes.c_int
    lib.muon_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double),
                                      ctypes.POINTER(ctypes.c_int64), ctypes.c_int]
    lib.muon_profile_read.restype = ctypes.c_int
    _lib = lib
    return lib


# ---- marshalling helpers ----------------------------------------------------------
def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return MUON_F32
    if t.dtype == torch.bfloat16:
        return MUON_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _shape3(t):
    if t.dim() == 2:
        return 1, t.shape[0], t.shape[1]
    if t.dim() == 3:
        return t.shape[0], t.shape[1], t.shape[2]
    raise ValueError("tensors must be [M,N] or [B,M,N]")


def _check_contig(*ts):
    for t in ts:
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous row-major")


def check(code: int, where: str) -> None:
    if code != MUON_OK:
        raise MuonError(code, where)


def make_config(steps: int = 5, coeffs: Optional[Sequence[Sequence[float]]] = None,
                a: float = 3.4445, b: float = -4.7750, c: float = 2.0315,
                eps: float = 1e-7, precision: int = NS_BF16):
    """Build an NsConfig; keeps the coefficient array alive on the object."""
    cfg = NsConfig()
    cfg.steps, cfg.a, cfg.b, cfg.c, cfg.eps, cfg.precision = steps, a, b, c, eps, precision
    if coeffs is not None:
        flat = [float(v) for row in coeffs for v in row]
        arr = (ctypes.c_float * max(1, len(flat)))(*flat)
        cfg.coeffs = ctypes.cast(arr, ctypes.POINTER(ctypes.c_float))
        cfg._keep = arr
    return cfg


# ---- entry points (same names as the C ABI) -------------------------------------------
def muon_ns_batched(X, steps: int = 5, a: float = 3.4445, b: float = -4.7750,
                    c: float = 2.0315, stream=None) -> None:
    """In-place NS of every [M,N] slice of a contiguous bf16 CUDA tensor."""
    _check_contig(X)
    B, M, N = _shape3(X)
    check(load().muon_ns_batched(X.data_ptr(), B, M, N, steps, a, b, c, _stream_ptr(stream)),
          "muon_ns_batched")


def muon_ns_batched_noalloc(X, steps: int = 5, a: float = 3.4445, b: float = -4.7750,
                            c: float = 2.0315, stream=None) -> None:
    """As muon_ns_batched, with the library's fixed workspace array (the call
    allocates no device memory)."""
    _check_contig(X)
    B, M, N = _shape3(X)
    check(load().muon_ns_batched_noalloc(X.data_ptr(), B, M, N, steps, a, b, c,
                                         _stream_ptr(stream)), "muon_ns_batched_noalloc")


def muon_ns_batched_ex(X, cfg=None, out=None, stream=None) -> None:
    """NS of every [M,N] slice of X (f32 or bf16) into X, or into `out`,
    which the library writes in X's dtype and shape (checked here: the C
    entry point sees only a pointer)."""
    _check_contig(X)
    B, M, N = _shape3(X)
    if out is not None:
        _check_contig(out)
        if out.dtype != X.dtype or tuple(out.shape) != tuple(X.shape):
            raise ValueError(f"out must match X: {out.dtype} {tuple(out.shape)} against "
                             f"{X.dtype} {tuple(X.shape)}")
    check(load().muon_ns_batched_ex(X.data_ptr(), _dtype_code(X), B, M, N,
                                    ctypes.byref(cfg) if cfg is not None else None,
                                    out.data_ptr() if out is not None else None,
                                    _stream_ptr(stream)), "muon_ns_batched_ex")


def make_groups(groups: Iterable[dict]):
    """[{"W","G","Mom"}] of contiguous CUDA tensors -> ctypes array."""
    groups = list(groups)
    arr = (Group * max(1, len(groups)))()
    for i, g in enumerate(groups):
        W, G, Mom = g["W"], g["G"], g["Mom"]
        _check_contig(W, G, Mom)
        B, M, N = _shape3(W)
        arr[i] = Group(W.data_ptr(), _dtype_code(W), G.data_ptr(), _dtype_code(G),
                       Mom.data_ptr(), B, M, N)
    return arr, len(groups)


def muon_step_grouped(groups, mu: float = 0.95, nesterov: bool = True, lr: float = 0.02,
                      wd: float = 0.01, scale_rule: int = SCALE_SQRT_MAX1_R_OVER_C,
                      ns_cfg=None, stream=None) -> None:
    """One fused Muon step over groups of [B,M,N] tensors (W, G, Mom)."""
    arr, n = groups if isinstance(groups, tuple) else make_groups(groups)
    lib = load()
    if ns_cfg is None:
        code = lib.muon_step_grouped(arr, n, mu, int(nesterov), lr, wd, scale_rule,
                                     _stream_ptr(stream))
    else:
        code = lib.muon_step_grouped_ex(arr, n, mu, int(nesterov), lr, wd, scale_rule,
                                        ctypes.byref(ns_cfg), _stream_ptr(stream))
    check(code, "muon_step_grouped")


muon_step_grouped_ex = muon_step_grouped


def muon_step_grouped_host(groups, mu: float = 0.95, nesterov: bool = True, lr: float = 0.02,
                           wd: float = 0.01, scale_rule: int = SCALE_SQRT_MAX1_R_OVER_C,
                           ns_cfg=None, stream=None) -> None:
    """One Muon step over groups of HOST (ideally pinned) [B,M,N] tensors; the
    library stages them through device memory.  Synchronise `stream` before
    reading the results."""
    arr, n = groups if isinstance(groups, tuple) else make_groups(groups)
    code = load().muon_step_grouped_host(arr, n, mu, int(nesterov), lr, wd, scale_rule,
                                         ctypes.byref(ns_cfg) if ns_cfg is not None else None,
                                         _stream_ptr(stream))
    check(code, "muon_step_grouped_host")


def muon_query_status(stream=None) -> int:
    return load().muon_query_status(_stream_ptr(stream))


def muon_debug_inject_stall(what: int) -> None:
    """Testing hook: the next launch of kind `what` (INJECT_GEMM or
    INJECT_SMALL) stalls on a wait nothing satisfies until its bound runs out."""
    check(load().muon_debug_inject_stall(int(what)), "muon_debug_inject_stall")


def muon_ns_path(rows: int, cols: int, cfg=None) -> int:
    """0 small-m kernel, 1 grouped GEMMs in X space, 2 grouped GEMMs in Gram
    space, for a stored [rows, cols] matrix (host-side decision)."""
    return load().muon_ns_path(rows, cols, ctypes.byref(cfg) if cfg is not None else None)


def muon_ns_gram_restart(m: int) -> int:
    """Restart period (NS steps) of the Gram-space path for small side m;
    0 = no restart."""
    return load().muon_ns_gram_restart(m)


def muon_debug_build() -> bool:
    """True for the -DMUON_DEBUG build (libmuon_debug.so)."""
    return bool(load().muon_debug_build())


def muon_debug_guard_check(stream=None) -> int:
    """Bytes found changed in the workspace guard bands since the last read
    (calls made with MUON_WS_GUARD=1); synchronises the stream."""
    bad = ctypes.c_int64(0)
    check(load().muon_debug_guard_check(_stream_ptr(stream), ctypes.byref(bad)),
          "muon_debug_guard_check")
    return bad.value


def muon_status_string(code: int) -> str:
    return load().muon_status_string(code).decode()


def muon_release_workspace() -> None:
    load().muon_release_workspace()


def muon_last_launch_count() -> int:
    return load().muon_last_launch_count()


def muon_profile_enable(enable: bool = True) -> int:
    return load().muon_profile_enable(int(enable))


def muon_profile_read():
    """{kind: (ms_total, launches)} since the last read (stream synchronised first)."""
    n = len(PROFILE_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    load().muon_profile_read(ms, cnt, n)
    return {k: (ms[i], cnt[i]) for i, k in enumerate(PROFILE_KINDS)}


def muon_adamw_grouped(groups, step: int, lr: float = 1e-3, betas=(0.9, 0.999),
                       eps: float = 1e-8, weight_decay: float = 0.01, stream=None) -> None:
    """One AdamW step over [{"param", "grad", "exp_avg", "exp_avg_sq"}] of
    contiguous CUDA tensors (any shape; fp32 state)."""
    groups = list(groups)
    arr = (AdamwGroup * max(1, len(groups)))()
    for i, g in enumerate(groups):
        p, gr, m, v = g["param"], g["grad"], g["exp_avg"], g["exp_avg_sq"]
        _check_contig(p, gr, m, v)
        arr[i] = AdamwGroup(p.data_ptr(), _dtype_code(p), gr.data_ptr(), _dtype_code(gr),
                            m.data_ptr(), v.data_ptr(), p.numel())
    cfg = AdamwConfig(lr, betas[0], betas[1], eps, weight_decay, step)
    check(load().muon_adamw_grouped(arr, len(groups), ctypes.byref(cfg), _stream_ptr(stream)),
          "muon_adamw_grouped")


def muon_ns_cost_table(shapes, cfg=None, reps: int = 5, stream=None):
    """Measured NS milliseconds per matrix for each (rows, cols) in `shapes`."""
    shapes = [(int(r), int(c)) for r, c in shapes]
    n = len(shapes)
    flat = (ctypes.c_int64 * max(1, 2 * n))(*[v for rc in shapes for v in rc])
    out = (ctypes.c_double * max(1, n))()
    check(load().muon_ns_cost_table(flat, n, ctypes.byref(cfg) if cfg is not None else None,
                                    reps, out, _stream_ptr(stream)), "muon_ns_cost_table")
    return [out[i] for i in range(n)]


def muon_assign_owners(costs, n_ranks: int, nbytes=None, elems=None, layers=None,
                       eps: float = 0.1):
    """Owner rank of each assignment unit (greedy LPT with a byte cap and
    layer spreading); host only."""
    n = len(costs)
    nbytes = nbytes if nbytes is not None else [0] * n
    elems = elems if elems is not None else [0] * n
    layers = layers if layers is not None else [-1] * n
    arr = (Unit * max(1, n))(*[Unit(float(costs[i]), int(nbytes[i]), int(elems[i]), int(layers[i]))
                               for i in range(n)])
    out = (ctypes.c_int32 * max(1, n))()
    check(load().muon_assign_owners(arr, n, n_ranks, eps, out), "muon_assign_owners")
    return [out[i] for i in range(n)]
