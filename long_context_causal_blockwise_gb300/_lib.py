"""ctypes binding of libattn.so (include/lcb_attn.h).

Argument marshalling only: torch tensors are passed as device pointers with
their strides, and the current CUDA stream is passed as the stream. Every step
of the computation runs in the library's CUDA kernels; if the library cannot be
loaded, every call raises (there is no fallback).
"""

import ctypes
import os

import torch

from . import build as _build

LCB_OK = 0
LCB_ERR_ARG = -1
LCB_ERR_UNSUPPORTED = -2
LCB_ERR_SCHEDULE = -3
LCB_ERR_CUDA = -4
LCB_ERR_TIMEOUT = -5
LCB_ERR_SCRATCH = -6
LCB_DTYPE_BF16 = 0
LCB_DTYPE_F32 = 1
LCB_OUT_F32_MERGE = 2
LCB_GRAD_BF16 = 0
LCB_GRAD_F32_ACCUM = 1
LCB_GRAD_F32_STORE = 2
TASK_DIAG, TASK_LOWER, TASK_UPPER, TASK_FULL, TASK_NONE = 0, 1, 2, 3, 4


class LcbTask(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("rank", "step", "src", "kind", "q_off", "q_len", "k_off", "k_len", "causal")]


class LcbFwdTask(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("q_off", "q_len", "k_off", "k_len", "causal", "o_dtype")]


class LcbBwdTask(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("q_off", "q_len", "k_off", "k_len", "causal")]


class AttnError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn} failed: {msg} ({status})")
        self.status = status


_LIB = None

_P, _I, _F, _LL, _SZ, _U64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong,
                               ctypes.c_size_t, ctypes.c_ulonglong)

_SIGNATURES = {
    "attn_status_string": ([_I], ctypes.c_char_p),
    "lcb_version": ([], _I),
    "attn_fwd": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P], _I),
    "attn_fwd_ex": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _LL, _LL, _LL, _LL, _LL, _LL, _I, _LL, _LL, _P],
                    _I),
    "attn_bwd_workspace_bytes": ([_I, _I, _I, _I], _SZ),
    "attn_bwd": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _SZ, _P], _I),
    "attn_bwd_preprocess": ([_P, _P, _P, _I, _I, _I, _I, _LL, _LL, _LL, _LL, _P], _I),
    "attn_bwd_ex": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _LL, _LL, _LL, _LL, _LL, _LL, _I,
                     _LL, _LL, _LL, _LL, _P], _I),
    "attn_bwd_fused_ex": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _LL, _LL, _LL, _LL, _LL,
                           _LL, _I, _LL, _LL, _LL, _LL, _P], _I),
    "attn_bwd_fused_group": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _LL, _LL, _LL, _LL, _LL,
                              _LL, _I, _LL, _LL, _LL, _LL, ctypes.POINTER(LcbBwdTask), _I, _P], _I),
    "lcb_dq_tiles_zero": ([_P, _LL, _P], _I),
    "lcb_dq_untile": ([_P, _LL, _LL, _P, _LL, _LL, _I, _I, _I, _P], _I),
    "attn_bwd_dkdv_ex": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _LL, _LL, _LL, _LL, _LL, _LL,
                          _I, _LL, _LL, _LL, _LL, _P], _I),
    "attn_bwd_dq_ex": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _LL, _LL, _LL, _LL, _LL, _LL, _I,
                        _LL, _LL, _LL, _LL, _P], _I),
    "attn_lse_merge": ([_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _LL, _LL, _LL, _LL, _LL, _LL, _LL, _LL, _P], _I),
    "attn_fwd_group": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _LL, _LL, _LL, _LL, _LL, _LL, _LL, _LL,
                        ctypes.POINTER(LcbFwdTask), _I, _P], _I),
    "zigzag_schedule": ([_I, _I, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(LcbTask)], _I),
    "ring_schedule": ([_I, _I, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(LcbTask)], _I),
    "lcb_cross_entropy": ([_P, _P, _P, _P, _P, _I, _I, _LL, _I, _I, _P], _I),
    "lcb_rope": ([_P, _P, _I, _I, _I, _I, ctypes.c_double, _LL, _I, _LL, _LL, _P], _I),
    "lcb_permute_rows": ([_P, _P, _P, _I, _LL, _P], _I),
    "lcb_scatter_rows": ([_P, _P, _P, _I, _LL, _P], _I),
    "lcb_cast_f32_bf16": ([_P, _P, _LL, _P], _I),
    "lcb_ulysses_all_to_all": ([_P, _P, _I, _I, _I, _I, _I, _I, _I, _P], _I),
    "lcb_set_wait_limit_ns": ([_U64], _U64),
    "attn_bwd_noalloc": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P], _I),
    "attn_bwd_noalloc_max_rows": ([], _LL),
    "lcb_selftest_bounded_wait": ([_P], _I),
    "lcb_take_device_status": ([ctypes.POINTER(ctypes.c_uint)], _I),
}

EXPORTED = tuple(_SIGNATURES)


def lib_path():
    return _build.LIB


def load(build_if_missing=True):
    """Loads (building first if needed) and returns the ctypes library."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.LIB
    if build_if_missing and (_build.needs_build()):
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"libattn.so not found at {path}; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, (args, res) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _LIB = lib
    return lib


def _check(fn, status):
    if status != LCB_OK:
        msg = load().attn_status_string(status).decode()
        raise AttnError(fn, status, msg)


def _stream(t):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name, ndim):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")
    if t.stride(-1) != 1:
        raise ValueError(f"{name} must be contiguous in its last dim")


def _bshd(t, name, dtype=torch.bfloat16):
    """(row_stride, batch_stride) of a [B,S,H,D] view whose [H,D] part is dense."""
    _need(t, dtype, name, 4)
    B, S, H, D = t.shape
    if t.stride(2) != D:
        raise ValueError(f"{name}: heads must be dense within a row")
    return t.stride(1), t.stride(0)


def _bhs(t, name):
    _need(t, torch.float32, name, 3)
    return t.stride(1), t.stride(0)


# ------------------------------------------------------------------ forward

def attn_fwd(q, k, v, causal=True, scale=None, o=None, lse=None):
    """Contiguous [B,S,H,D] bf16 forward; returns (o bf16, lse fp32 [B,H,S])."""
    B, S, H, D = q.shape
    scale = D ** -0.5 if scale is None else scale
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _need(t, torch.bfloat16, n, 4)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous (use attn_fwd_ex for strided views)")
    if not lse.is_contiguous():
        raise ValueError("lse must be contiguous")
    _check("attn_fwd", load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, S, D, int(causal),
                                       float(scale), _stream(q)))
    return o, lse


def attn_fwd_ex(q, k, v, o, lse, causal, scale, merge=False):
    """Forward on strided [B,S,H,D] views; o bf16 or fp32; lse [B,H,Sq] view.

    merge=True: o (fp32) and lse hold a partial result over other keys and this
    block is merged into them in the kernel (a fused ring step)."""
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    qr, qb = _bshd(q, "q")
    kr, kb = _bshd(k, "k")
    vr, vb = _bshd(v, "v")
    if (vr, vb) != (kr, kb):
        raise ValueError("k and v must share strides")
    o_dtype = LCB_DTYPE_F32 if o.dtype == torch.float32 else LCB_DTYPE_BF16
    if merge:
        if o.dtype != torch.float32:
            raise ValueError("merge mode needs an fp32 accumulator")
        o_dtype = LCB_OUT_F32_MERGE
    orr, ob = _bshd(o, "o", o.dtype)
    lh, lb = _bhs(lse, "lse")
    _check("attn_fwd_ex", load().attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Sq, Sk, D,
                                             int(causal), float(scale), qr, qb, kr, kb, orr, ob, o_dtype, lh, lb,
                                             _stream(q)))
    return o, lse


_OUT_MODES = {"bf16": LCB_DTYPE_BF16, "f32": LCB_DTYPE_F32, "merge": LCB_OUT_F32_MERGE}


def attn_fwd_group(q, k, v, o, lse, tasks, scale):
    """Several forward blocks over shared [B,S,H,D] views in one launch.

    tasks: sequence of (q_off, q_len, k_off, k_len, causal, out) with out one
    of "bf16", "f32", "merge" (o's dtype: bf16 for "bf16", fp32 otherwise);
    query ranges must not overlap."""
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    qr, qb = _bshd(q, "q")
    kr, kb = _bshd(k, "k")
    if _bshd(v, "v") != (kr, kb):
        raise ValueError("k and v must share strides")
    orr, ob = _bshd(o, "o", o.dtype)
    lh, lb = _bhs(lse, "lse")
    arr = (LcbFwdTask * max(1, len(tasks)))()
    for i, (qo, ql, ko, kl, causal, out) in enumerate(tasks):
        want = torch.bfloat16 if out == "bf16" else torch.float32
        if o.dtype != want:
            raise ValueError(f"task output {out!r} needs o of dtype {want}")
        arr[i] = LcbFwdTask(int(qo), int(ql), int(ko), int(kl), int(causal), _OUT_MODES[out])
    _check("attn_fwd_group", load().attn_fwd_group(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Sq, Sk, D,
                                                   float(scale), qr, qb, kr, kb, orr, ob, lh, lb, arr, len(tasks),
                                                   _stream(q)))
    return o, lse


# ------------------------------------------------------------------ backward

def attn_bwd_workspace_bytes(B, H, S, D=128):
    return int(load().attn_bwd_workspace_bytes(B, H, S, D))


def attn_bwd(q, k, v, o, lse, do, causal=True, scale=None, dq=None, dk=None, dv=None, workspace=None):
    """Contiguous backward; returns (dq, dk, dv) bf16."""
    B, S, H, D = q.shape
    scale = D ** -0.5 if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _need(t, torch.bfloat16, n, 4)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    ws_bytes = attn_bwd_workspace_bytes(B, H, S, D)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    _check("attn_bwd", load().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk),
                                       _ptr(dv), B, H, S, D, int(causal), float(scale), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(q)))
    return dq, dk, dv


def attn_bwd_noalloc(q, k, v, o, lse, do, causal=True, scale=None, dq=None, dk=None, dv=None):
    """attn_bwd without a workspace: Delta lives in the library's fixed device array.

    For callers that cannot allocate device memory (see include/lcb_attn.h);
    B*H*S must not exceed attn_bwd_noalloc_max_rows()."""
    B, S, H, D = q.shape
    scale = D ** -0.5 if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _need(t, torch.bfloat16, n, 4)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    _check("attn_bwd_noalloc", load().attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                                       _ptr(dq), _ptr(dk), _ptr(dv), B, H, S, D, int(causal),
                                                       float(scale), _stream(q)))
    return dq, dk, dv


def attn_bwd_noalloc_max_rows():
    return int(load().attn_bwd_noalloc_max_rows())


def attn_bwd_preprocess(o, do, delta):
    B, S, H, D = o.shape
    r, b = _bshd(o, "o")
    if _bshd(do, "do") != (r, b):
        raise ValueError("o and do must share strides")
    dh, db = _bhs(delta, "delta")
    _check("attn_bwd_preprocess", load().attn_bwd_preprocess(_ptr(o), _ptr(do), _ptr(delta), B, H, S, D, r, b, dh,
                                                             db, _stream(o)))
    return delta


def attn_bwd_ex(q, k, v, lse, delta, do, dq, dk, dv, causal, scale, accumulate=True, passes="both"):
    """Block backward with given row statistics.

    bf16 gradients are overwritten; fp32 gradients are accumulated into
    (accumulate=True) or overwritten (accumulate=False).
    passes: "both" (the deterministic two-pass form), "dkdv" or "dq" (one of
    its passes), or "fused" (one pass; dq is then a tiled fp32 accumulator
    [B, H, T, 16384] from dq_tiles_zeros, or a slice of one along T starting
    at this call's first query tile, always added into; dk/dv follow their
    dtype and `accumulate`)."""
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    qr, qb = _bshd(q, "q")
    if _bshd(do, "do") != (qr, qb):
        raise ValueError("q and do must share strides")
    kr, kb = _bshd(k, "k")
    if _bshd(v, "v") != (kr, kb):
        raise ValueError("k and v must share strides")
    lh, lb = _bhs(lse, "lse")
    if _bhs(delta, "delta") != (lh, lb):
        raise ValueError("lse and delta must share strides")
    gdt = dk.dtype
    if dv.dtype != gdt:
        raise ValueError("dk and dv must share a dtype")
    if passes == "fused":
        if dq.dtype != torch.float32 or dq.dim() != 4 or dq.shape[3] != 128 * 128 or dq.stride(3) != 1 \
                or dq.stride(2) != 128 * 128 or dq.shape[0] != B or dq.shape[1] != H or dq.shape[2] * 128 < Sq:
            raise ValueError("the fused pass adds dQ into a tiled fp32 accumulator (dq_tiles_zeros)")
    elif dq.dtype != gdt:
        raise ValueError("dq, dk, dv must share a dtype")
    if gdt == torch.float32:
        grad_mode = LCB_GRAD_F32_ACCUM if accumulate else LCB_GRAD_F32_STORE
    else:
        grad_mode = LCB_GRAD_BF16
    if passes == "fused":
        dqr, dqb = dq.stride(1), dq.stride(0)  # tile head and batch strides
    else:
        dqr, dqb = _bshd(dq, "dq", dq.dtype)
    dkr, dkb = _bshd(dk, "dk", gdt)
    if _bshd(dv, "dv", gdt) != (dkr, dkb):
        raise ValueError("dk and dv must share strides")
    fname = {"both": "attn_bwd_ex", "dkdv": "attn_bwd_dkdv_ex", "dq": "attn_bwd_dq_ex",
             "fused": "attn_bwd_fused_ex"}[passes]
    _check(fname, getattr(load(), fname)(_ptr(q), _ptr(k), _ptr(v), _ptr(lse), _ptr(delta), _ptr(do), _ptr(dq),
                                             _ptr(dk), _ptr(dv), B, H, Sq, Sk, D, int(causal), float(scale), qr, qb,
                                             kr, kb, lh, lb, grad_mode, dqr, dqb, dkr, dkb, _stream(q)))
    return dq, dk, dv


def attn_bwd_group(q, k, v, lse, delta, do, dq_tiles, dk, dv, tasks, scale, accumulate=True):
    """Several one-pass backward blocks over shared [B,S,H,D] views in one launch.

    tasks: sequence of (q_off, q_len, k_off, k_len, causal), q_off a multiple
    of 128, key ranges disjoint. dq_tiles: the tiled accumulator of all of q's
    rows (dq_tiles_zeros), added into; dk/dv as in attn_bwd_ex(passes="fused")."""
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    qr, qb = _bshd(q, "q")
    if _bshd(do, "do") != (qr, qb):
        raise ValueError("q and do must share strides")
    kr, kb = _bshd(k, "k")
    if _bshd(v, "v") != (kr, kb):
        raise ValueError("k and v must share strides")
    lh, lb = _bhs(lse, "lse")
    if _bhs(delta, "delta") != (lh, lb):
        raise ValueError("lse and delta must share strides")
    if dq_tiles.dtype != torch.float32 or dq_tiles.dim() != 4 or dq_tiles.shape[:2] != (B, H) \
            or dq_tiles.shape[2] * 128 < Sq or dq_tiles.stride(3) != 1 or dq_tiles.stride(2) != 128 * 128:
        raise ValueError("dq_tiles must be a tiled fp32 accumulator covering q (dq_tiles_zeros)")
    gdt = dk.dtype
    if dv.dtype != gdt:
        raise ValueError("dk and dv must share a dtype")
    if gdt == torch.float32:
        grad_mode = LCB_GRAD_F32_ACCUM if accumulate else LCB_GRAD_F32_STORE
    else:
        grad_mode = LCB_GRAD_BF16
    dkr, dkb = _bshd(dk, "dk", gdt)
    if _bshd(dv, "dv", gdt) != (dkr, dkb):
        raise ValueError("dk and dv must share strides")
    arr = (LcbBwdTask * max(1, len(tasks)))(*[LcbBwdTask(*(int(x) for x in t)) for t in tasks])
    _check("attn_bwd_fused_group", load().attn_bwd_fused_group(
        _ptr(q), _ptr(k), _ptr(v), _ptr(lse), _ptr(delta), _ptr(do), _ptr(dq_tiles), _ptr(dk), _ptr(dv), B, H, Sq,
        Sk, D, float(scale), qr, qb, kr, kb, lh, lb, grad_mode, dq_tiles.stride(1), dq_tiles.stride(0), dkr, dkb, arr,
        len(tasks), _stream(q)))
    return dq_tiles, dk, dv


def dq_tiles_zeros(B, H, S, device):
    """A zeroed tiled fp32 dQ accumulator for the fused pass: [B, H, ceil(S/128), 128*128]."""
    return torch.zeros((B, H, (S + 127) // 128, 128 * 128), dtype=torch.float32, device=device)


def dq_tiles_zero_(tiles):
    """Zeroes a tiled dQ accumulator in place (on the current stream); returns it."""
    if tiles.dtype != torch.float32 or not tiles.is_contiguous():
        raise ValueError("tiles must be a contiguous fp32 accumulator (dq_tiles_zeros)")
    _check("lcb_dq_tiles_zero", load().lcb_dq_tiles_zero(_ptr(tiles), tiles.numel(), _stream(tiles)))
    return tiles


def dq_untile(tiles, dq):
    """Tiled fp32 accumulator -> bf16 rows of dq ([B, S, H, D] view); returns dq."""
    B, S, H, D = dq.shape
    r, b = _bshd(dq, "dq")
    if tiles.dtype != torch.float32 or tiles.dim() != 4 or tiles.shape[:2] != (B, H) or tiles.shape[2] * 128 < S \
            or tiles.stride(3) != 1 or tiles.stride(2) != 128 * 128:
        raise ValueError("tiles must be a tiled fp32 accumulator covering dq (dq_tiles_zeros)")
    _check("lcb_dq_untile", load().lcb_dq_untile(_ptr(tiles), tiles.stride(1), tiles.stride(0), _ptr(dq), r, b, B, H,
                                                 S, _stream(dq)))
    return dq


# ------------------------------------------------------------------ merge / zigzag

def attn_lse_merge(o_acc, lse_acc, o_b, lse_b, o_out_bf16=None):
    """In-place (o_acc fp32, lse_acc) <- merge with (o_b bf16/fp32, lse_b)."""
    B, R, H, D = o_acc.shape
    if o_b.shape != o_acc.shape or lse_b.shape != lse_acc.shape:
        raise ValueError("merge operands must have matching shapes")
    r, b = _bshd(o_acc, "o_acc", torch.float32)
    rb, bb = _bshd(o_b, "o_b", o_b.dtype)
    lh, lb = _bhs(lse_acc, "lse_acc")
    lbh, lbb = _bhs(lse_b, "lse_b")
    if o_out_bf16 is not None and _bshd(o_out_bf16, "o_out_bf16") != (r, b):
        raise ValueError("o_out_bf16 must share o_acc's strides")
    odt = LCB_DTYPE_F32 if o_b.dtype == torch.float32 else LCB_DTYPE_BF16
    _check("attn_lse_merge", load().attn_lse_merge(_ptr(o_acc), _ptr(lse_acc), _ptr(o_b), _ptr(lse_b), odt,
                                                   None if o_out_bf16 is None else _ptr(o_out_bf16), B, H, R, D, r,
                                                   b, rb, bb, lh, lb, lbh, lbb, _stream(o_acc)))
    return o_acc, lse_acc


def zigzag_schedule(S, P):
    """Host call: returns (perm list[int], tasks list[dict])."""
    perm = (ctypes.c_int * S)()
    tasks = (LcbTask * (P * P))()
    _check("zigzag_schedule", load().zigzag_schedule(S, P, perm, tasks))
    return list(perm), [{f: getattr(t, f) for f, _ in LcbTask._fields_} for t in tasks]


def ring_schedule(S, P):
    """Host call: the plain (contiguous) ring; returns (perm list[int], tasks list[dict])."""
    perm = (ctypes.c_int * S)()
    tasks = (LcbTask * (P * P))()
    _check("ring_schedule", load().ring_schedule(S, P, perm, tasks))
    return list(perm), [{f: getattr(t, f) for f, _ in LcbTask._fields_} for t in tasks]


_CE_MODES = {"fwd": 0, "fwd_bwd": 1, "bwd": 2}


def cross_entropy(logits, labels, ignore_index=-100, mode="fwd_bwd", dloss=None, lse=None, loss=None):
    """Cross-entropy of bf16 logits [N, V] against int64 labels [N].

    mode "fwd": returns (loss, lse); "fwd_bwd": also overwrites logits with
    dloss_i * (softmax - onehot) (dloss None: 1 per row); "bwd": the gradient
    alone from a given lse. Returns (loss, lse)."""
    if logits.dim() != 2 or logits.dtype != torch.bfloat16 or logits.stride(1) != 1:
        raise ValueError("logits must be a bf16 [N, V] view with unit column stride")
    N, V = logits.shape
    if labels.dtype != torch.int64 or labels.shape != (N,) or not labels.is_contiguous():
        raise ValueError("labels must be a contiguous int64 [N] tensor")
    dev = logits.device
    if mode == "bwd":
        if lse is None:
            raise ValueError("mode 'bwd' needs the lse of a previous forward")
    else:
        lse = torch.empty(N, dtype=torch.float32, device=dev) if lse is None else lse
        loss = torch.empty(N, dtype=torch.float32, device=dev) if loss is None else loss
    for t, n in ((lse, "lse"), (loss, "loss"), (dloss, "dloss")):
        if t is not None and (t.dtype != torch.float32 or t.shape != (N,) or not t.is_contiguous()):
            raise ValueError(f"{n} must be a contiguous fp32 [N] tensor")
    _check("lcb_cross_entropy", load().lcb_cross_entropy(
        _ptr(logits), _ptr(labels), None if loss is None else _ptr(loss), _ptr(lse),
        None if dloss is None else _ptr(dloss), N, V, logits.stride(0), int(ignore_index), _CE_MODES[mode],
        _stream(logits)))
    return loss, lse


def rope(x, theta, pos0=0, inverse=False, out=None):
    """RoPE (raised base theta) of a bf16 [B, S, H, 128] view; out=None rotates in place.

    inverse=True applies the transpose (maps dQ/dK of rotated inputs back)."""
    B, S, H, D = x.shape
    out = x if out is None else out
    r, b = _bshd(x, "x")
    if _bshd(out, "out") != (r, b):
        raise ValueError("x and out must share strides")
    _check("lcb_rope", load().lcb_rope(_ptr(x), _ptr(out), B, S, H, D, float(theta), int(pos0), int(inverse), r, b,
                                       _stream(x)))
    return out


def permute_rows(src, dst, perm_dev, scatter=False):
    """Rows of contiguous [1, S, ...] tensors: dst[t] = src[perm[t]] (or the scatter)."""
    if not (src.is_contiguous() and dst.is_contiguous()) or src.shape != dst.shape or src.dtype != dst.dtype:
        raise ValueError("src and dst must be contiguous tensors of one shape and dtype")
    if perm_dev.dtype != torch.int32 or not perm_dev.is_cuda:
        raise ValueError("perm must be a CUDA int32 tensor")
    rows = perm_dev.numel()
    row_bytes = src.numel() // rows * src.element_size()
    fn = load().lcb_scatter_rows if scatter else load().lcb_permute_rows
    _check("permute_rows", fn(_ptr(src), _ptr(dst), _ptr(perm_dev), rows, row_bytes, _stream(src)))
    return dst


ULYSSES_SEQ_TO_HEAD, ULYSSES_HEAD_TO_SEQ = 0, 1


def ulysses_all_to_all(src, P, to_heads=True, out=None):
    """The Ulysses all-to-all of P emulated ranks (include/lcb_attn.h).

    to_heads=True: src is a contiguous [B, S, H, D] tensor (the ranks'
    sequence pieces); returns the head layout as a [P*B, S, H/P, D] tensor
    (rank j's part is rows [j*B, (j+1)*B) of dim 0). to_heads=False: the
    inverse; src is [P*B, S, H/P, D] and the result [B, S, H, D]."""
    if not src.is_cuda or not src.is_contiguous() or src.dim() != 4:
        raise ValueError("src must be a contiguous 4-d CUDA tensor")
    if src.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("src must be bf16 or fp32")
    if to_heads:
        B, S, H, D = src.shape
        if H % P:
            raise ValueError("P must divide H")
        shape = (P * B, S, H // P, D)
    else:
        PB, S, Hp, D = src.shape
        if PB % P:
            raise ValueError("dim 0 of a head-layout tensor is P*B")
        B, H = PB // P, Hp * P
        shape = (B, S, H, D)
    if out is None:
        out = torch.empty(shape, dtype=src.dtype, device=src.device)
    elif tuple(out.shape) != shape or out.dtype != src.dtype or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous {shape} tensor of src's dtype")
    _check("lcb_ulysses_all_to_all", load().lcb_ulysses_all_to_all(
        _ptr(src), _ptr(out), B, S, H, D, P, src.element_size(),
        ULYSSES_SEQ_TO_HEAD if to_heads else ULYSSES_HEAD_TO_SEQ, _stream(src)))
    return out


def cast_f32_bf16(src, dst):
    if src.dtype != torch.float32 or dst.dtype != torch.bfloat16 or src.numel() != dst.numel():
        raise ValueError("cast_f32_bf16 wants fp32 src and bf16 dst of one size")
    if not (src.is_contiguous() and dst.is_contiguous()):
        raise ValueError("cast_f32_bf16 wants contiguous tensors")
    _check("lcb_cast_f32_bf16", load().lcb_cast_f32_bf16(_ptr(src), _ptr(dst), src.numel(), _stream(src)))
    return dst


def set_wait_limit_ns(ns):
    return int(load().lcb_set_wait_limit_ns(int(ns)))


def selftest_bounded_wait():
    return int(load().lcb_selftest_bounded_wait(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))


def take_device_status():
    where = ctypes.c_uint(0)
    bits = load().lcb_take_device_status(ctypes.byref(where))
    return int(bits), int(where.value)
