"""Thin Python binding of the KDA C ABI (``include/kda.h``).

Argument marshalling only: every step of the operator runs in the CUDA kernels
of ``_build/libkda.so``.  Tensors are torch CUDA tensors (PyTorch supplies the
device memory and the stream); their data pointers are handed to the C entry
points.  If the library has not been built this module raises on first use --
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkda.so")

KDA_BF16, KDA_F32 = 0, 1
STATUS = {0: "KDA_OK", 1: "KDA_ERR_NULL", 2: "KDA_ERR_SHAPE", 3: "KDA_ERR_DTYPE",
          4: "KDA_ERR_ALIGN", 5: "KDA_ERR_SEQLENS", 6: "KDA_ERR_UNSUPPORTED",
          7: "KDA_ERR_CUDA", 8: "KDA_ERR_WORKSPACE", 9: "KDA_ERR_TIMEOUT"}
KDA_OK, KDA_ERR_TIMEOUT = 0, 9
WAIT_LIMIT_DEFAULT = 0xFFFFFFFF

EXPORTED = ["kda_prefill", "kda_prefill_recurrent", "kda_prefill_workspace_size",
            "kda_decode_step", "kda_gate_norm", "kda_status_str", "kda_last_error_string",
            "kda_version", "kda_launch_count", "kda_prefill_noalloc", "kda_prefill_snapshot_count",
            "kda_short_conv", "kda_short_conv_step", "kda_kcp_apply", "kda_prefill_records",
            "kda_prefill_scan", "kda_get_last_device_error", "kda_debug_set_wait_limit",
            "kda_prefill_from_host", "kda_prefill_from_host_staging_size"]

_vp = ctypes.c_void_p


class PrefillArgs(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int), ("T_total", ctypes.c_int),
        ("H", ctypes.c_int), ("dk", ctypes.c_int), ("dv", ctypes.c_int),
        ("qkv_dtype", ctypes.c_int),
        ("cu_seqlens", _vp), ("cu_seqlens_host", _vp),
        ("q", _vp), ("k", _vp), ("v", _vp), ("z", _vp), ("beta", _vp), ("A", _vp),
        ("g_min", ctypes.c_float), ("scale", ctypes.c_float), ("qk_l2norm", ctypes.c_int),
        ("S0", _vp), ("o", _vp), ("S_T", _vp),
        ("g_in", _vp), ("norm_w", _vp), ("norm_eps", ctypes.c_float), ("y", _vp),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
        ("snap_interval", ctypes.c_int), ("S_snap", _vp), ("gate_mode", ctypes.c_int),
    ]


class DecodeArgs(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int), ("H", ctypes.c_int), ("dk", ctypes.c_int), ("dv", ctypes.c_int),
        ("num_slots", ctypes.c_int),
        ("q", _vp), ("k", _vp), ("v", _vp), ("z", _vp), ("beta", _vp), ("A", _vp),
        ("g_min", ctypes.c_float), ("scale", ctypes.c_float), ("qk_l2norm", ctypes.c_int),
        ("state", _vp), ("slots", _vp), ("o", _vp),
        ("g_in", _vp), ("norm_w", _vp), ("norm_eps", ctypes.c_float), ("y", _vp),
        ("gate_mode", ctypes.c_int),
    ]


GATES = {"bounded": 0, "softplus": 1}   # kda_gate: K3's bounded gate, Kimi Linear's Softplus gate


class ShortConvArgs(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int), ("T_total", ctypes.c_int), ("channels", ctypes.c_int),
        ("width", ctypes.c_int), ("dtype", ctypes.c_int),
        ("cu_seqlens", _vp), ("cu_seqlens_host", _vp),
        ("x", _vp), ("weight", _vp), ("bias", _vp), ("state_in", _vp), ("state_out", _vp),
        ("y", _vp), ("activation", ctypes.c_int),
    ]


class ShortConvStepArgs(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int), ("channels", ctypes.c_int), ("width", ctypes.c_int), ("num_slots", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("x", _vp), ("weight", _vp), ("bias", _vp), ("state", _vp), ("slots", _vp),
        ("y", _vp), ("activation", ctypes.c_int),
    ]


class KDAError(RuntimeError):
    pass


_lib = None


def load_library(path: str = LIB_PATH):
    """Load the compiled library (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"KDA CUDA library not built: {path} is missing "
                          "(run serving_kda_chunked_gated_gb300.build.build())")
    lib = ctypes.CDLL(path)
    lib.kda_prefill.argtypes = [ctypes.POINTER(PrefillArgs), _vp]
    lib.kda_prefill.restype = ctypes.c_int
    lib.kda_prefill_records.argtypes = [ctypes.POINTER(PrefillArgs), _vp]
    lib.kda_prefill_records.restype = ctypes.c_int
    lib.kda_prefill_scan.argtypes = [ctypes.POINTER(PrefillArgs), ctypes.c_int, _vp]
    lib.kda_prefill_scan.restype = ctypes.c_int
    lib.kda_prefill_noalloc.argtypes = [ctypes.POINTER(PrefillArgs), _vp]
    lib.kda_prefill_noalloc.restype = ctypes.c_int
    lib.kda_prefill_recurrent.argtypes = [ctypes.POINTER(PrefillArgs), _vp]
    lib.kda_prefill_recurrent.restype = ctypes.c_int
    lib.kda_prefill_workspace_size.argtypes = [ctypes.POINTER(PrefillArgs)]
    lib.kda_prefill_workspace_size.restype = ctypes.c_size_t
    lib.kda_prefill_snapshot_count.argtypes = [ctypes.POINTER(PrefillArgs)]
    lib.kda_prefill_snapshot_count.restype = ctypes.c_long
    lib.kda_decode_step.argtypes = [ctypes.POINTER(DecodeArgs), _vp]
    lib.kda_kcp_apply.restype = ctypes.c_int
    lib.kda_kcp_apply.argtypes = [_vp, _vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp]
    lib.kda_short_conv.restype = ctypes.c_int
    lib.kda_short_conv.argtypes = [ctypes.POINTER(ShortConvArgs), _vp]
    lib.kda_short_conv_step.restype = ctypes.c_int
    lib.kda_short_conv_step.argtypes = [ctypes.POINTER(ShortConvStepArgs), _vp]
    lib.kda_decode_step.restype = ctypes.c_int
    lib.kda_gate_norm.argtypes = [_vp, _vp, _vp, ctypes.c_float, _vp, ctypes.c_long,
                                  ctypes.c_int, ctypes.c_int, _vp]
    lib.kda_gate_norm.restype = ctypes.c_int
    lib.kda_status_str.argtypes = [ctypes.c_int]
    lib.kda_status_str.restype = ctypes.c_char_p
    lib.kda_last_error_string.restype = ctypes.c_char_p
    lib.kda_version.restype = ctypes.c_char_p
    lib.kda_launch_count.restype = ctypes.c_uint64
    lib.kda_get_last_device_error.argtypes = [_vp, _vp]
    lib.kda_get_last_device_error.restype = ctypes.c_int
    lib.kda_debug_set_wait_limit.argtypes = [ctypes.c_uint32]
    lib.kda_prefill_from_host.argtypes = [ctypes.POINTER(PrefillArgs), ctypes.c_int, _vp, ctypes.c_size_t, _vp]
    lib.kda_prefill_from_host.restype = ctypes.c_int
    lib.kda_prefill_from_host_staging_size.argtypes = [ctypes.POINTER(PrefillArgs), ctypes.c_int]
    lib.kda_prefill_from_host_staging_size.restype = ctypes.c_size_t
    lib.kda_debug_set_wait_limit.restype = ctypes.c_uint32
    _lib = lib
    return lib


def launch_count() -> int:
    """Kernel launches enqueued by this library from the calling thread so far."""
    return int(load_library().kda_launch_count())


def device_error(workspace=None, stream=None) -> int:
    """``kda_get_last_device_error``: waits for ``stream``, then reads and clears
    the error word of ``workspace`` (a prefill workspace tensor), or of the
    array ``kda_prefill_noalloc`` uses when ``workspace`` is None.  Returns
    KDA_OK (0) or KDA_ERR_TIMEOUT (9); raises on any other status."""
    st = load_library().kda_get_last_device_error(_p(workspace), _stream(stream))
    if st not in (KDA_OK, KDA_ERR_TIMEOUT):
        _check(st, "kda_get_last_device_error")
    return st


def set_wait_limit(polls: int) -> int:
    """``kda_debug_set_wait_limit`` (test hook): the poll bound of the prefill
    kernels' waits on copies and MMAs for later launches; WAIT_LIMIT_DEFAULT
    restores the default, 0 makes every such wait give up at once.  Returns the
    previous setting."""
    return int(load_library().kda_debug_set_wait_limit(ctypes.c_uint32(polls)))


def _check(status: int, what: str):
    if status != 0:
        lib = load_library()
        msg = lib.kda_status_str(status).decode()
        if status == 7:
            msg += ": " + lib.kda_last_error_string().decode()
        raise KDAError(f"{what} failed with {STATUS.get(status, status)} ({msg})")


def _p(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise KDAError(f"unsupported dtype {t.dtype}")


def make_prefill_args(q, k, v, z, beta, A, cu_seqlens, cu_seqlens_host, o, S0=None, S_T=None,
                      g_in=None, norm_w=None, y=None, g_min=-5.0, scale=1.0, qk_l2norm=True,
                      norm_eps=1e-6, workspace=None, gate="bounded") -> PrefillArgs:
    """Fill the C argument struct from tensors (no validation beyond dtype mapping)."""
    T, H, dk = q.shape
    dv = v.shape[2]
    cu_host = cu_seqlens_host
    a = PrefillArgs()
    a.num_seqs = int(cu_host.numel() - 1)
    a.T_total, a.H, a.dk, a.dv = int(T), int(H), int(dk), int(dv)
    a.qkv_dtype = _dtype_code(q)
    a.cu_seqlens = cu_seqlens.data_ptr()
    a.cu_seqlens_host = cu_host.data_ptr()
    for name, t in (("q", q), ("k", k), ("v", v), ("z", z), ("beta", beta), ("A", A),
                    ("S0", S0), ("o", o), ("S_T", S_T), ("g_in", g_in), ("norm_w", norm_w),
                    ("y", y)):
        setattr(a, name, t.data_ptr() if t is not None else None)
    a.g_min, a.scale, a.qk_l2norm, a.norm_eps = float(g_min), float(scale), int(bool(qk_l2norm)), float(norm_eps)
    a.gate_mode = GATES[gate]
    if workspace is not None:
        a.workspace = workspace.data_ptr()
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    return a


def prefill_noalloc_raw(args: PrefillArgs, stream=None):
    """``kda_prefill_noalloc``: for callers that cannot allocate device memory.
    The workspace fields of ``args`` are ignored; the library's fixed device
    scratch array is used instead.  Calls on unordered streams race on it."""
    _check(load_library().kda_prefill_noalloc(ctypes.byref(args), _stream(stream)), "kda_prefill_noalloc")


def prefill_workspace_size(args: PrefillArgs) -> int:
    return int(load_library().kda_prefill_workspace_size(ctypes.byref(args)))


def prefill_raw(args: PrefillArgs, stream=None, recurrent: bool = False):
    lib = load_library()
    fn = lib.kda_prefill_recurrent if recurrent else lib.kda_prefill
    _check(fn(ctypes.byref(args), _stream(stream)), "kda_prefill_recurrent" if recurrent else "kda_prefill")


PREFILL_MIN_WORKSPACE = 256   # smallest workspace of the tensor-core path (single-pass schedule)
_WS_CACHE = {}                # prefill(workspace="cache"): one buffer per device


def cached_workspace(dev):
    """The buffer ``prefill(workspace="cache")`` uses on ``dev`` (None before the
    first such call)."""
    dev = torch.device(dev)
    return _WS_CACHE.get((dev.type, dev.index if dev.index is not None else torch.cuda.current_device()))


def release_workspace_cache():
    """Drop the cached workspaces (their memory returns to torch's allocator)."""
    _WS_CACHE.clear()


_STAGING = {}                 # prefill_from_host: one staging buffer per device


def prefill_from_host(q, k, v, z, beta, A, S0=None, g_in=None, norm_w=None, out=None, slab=16384,
                      g_min=-5.0, scale=1.0, qk_l2norm=True, norm_eps=1e-6, gate="bounded", stream=None):
    """KDA prefill of one sequence held in (pinned) host memory, results back to
    host memory, through ``kda_prefill_from_host``: the library cuts the sequence
    into slabs of ``slab`` tokens (a multiple of 64) and overlaps the copies with
    the compute.  q, k, v, g_in [T, H, d] bf16 (or f32), z [T, H, d] f32, beta
    [T, H], A [H], S0 [1, H, d, d] or None, all host tensors; out = (o, y, S_T)
    host tensors (y None without g_in), allocated pinned when None.  The device
    staging comes from a per-device cache.  Returns (o, S_T, y) on the host
    once the call's stream has completed.
    """
    T, H, d = q.shape
    dv = v.shape[2]
    dev = torch.device("cuda", torch.cuda.current_device())
    gate_on = g_in is not None
    if out is None:
        out = (torch.empty((T, H, dv), dtype=q.dtype).pin_memory(),
               torch.empty((T, H, dv), dtype=torch.bfloat16).pin_memory() if gate_on else None,
               torch.empty((1, H, d, dv), dtype=torch.float32).pin_memory())
    o_h, y_h, S_h = out
    a = PrefillArgs()
    a.num_seqs, a.T_total, a.H, a.dk, a.dv = 1, int(T), int(H), int(d), int(dv)
    a.qkv_dtype = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("z", z), ("beta", beta), ("A", A), ("S0", S0),
                    ("o", o_h), ("S_T", S_h), ("g_in", g_in), ("norm_w", norm_w), ("y", y_h)):
        setattr(a, name, t.data_ptr() if t is not None else None)
    a.g_min, a.scale, a.qk_l2norm, a.norm_eps = float(g_min), float(scale), int(bool(qk_l2norm)), float(norm_eps)
    a.gate_mode = GATES[gate]
    lib = load_library()
    need = int(lib.kda_prefill_from_host_staging_size(ctypes.byref(a), int(slab)))
    if need == 0:
        raise ValueError("kda_prefill_from_host: unsupported slab or shape")
    key = (dev.type, dev.index)
    st = _STAGING.get(key)
    if st is None or st.numel() < need:
        _STAGING[key] = st = torch.empty(need, dtype=torch.uint8, device=dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    _check(lib.kda_prefill_from_host(ctypes.byref(a), int(slab), st.data_ptr(), st.numel(), _stream(s)),
           "kda_prefill_from_host")
    return o_h, S_h, y_h


def snapshot_count(cu_seqlens_host, interval: int) -> int:
    """Rows of the snapshot output for packed sequences (see kda.h)."""
    cu = [int(x) for x in cu_seqlens_host]
    return sum((cu[i + 1] - cu[i]) // interval for i in range(len(cu) - 1))


def prefill(q, k, v, z, beta, A, cu_seqlens=None, S0=None, g_in=None, norm_w=None,
            g_min=-5.0, scale=1.0, qk_l2norm=True, norm_eps=1e-6, want_state=True,
            out=None, stream=None, recurrent=False, workspace=None, snap_interval=0, gate="bounded",
            want_o=True):
    """KDA chunked prefill through ``kda_prefill``.

    q, k, z: [T, H, dk]; v: [T, H, dv]; beta: [T, H]; A: [H]; cu_seqlens: int32
    [N+1] on the device (None = one sequence).  Returns (o, S_T, y), or
    (o, S_T, y, S_snap) when snap_interval > 0 (prefix-cache snapshots).
    """
    T, H, dk = q.shape
    dv = v.shape[2]
    dev = q.device
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=dev)
    cu_host = cu_seqlens.to("cpu")
    N = cu_host.numel() - 1
    o = (out["o"] if out else torch.empty((T, H, dv), dtype=q.dtype, device=dev)) if want_o else None
    S_T = (out["S_T"] if out else torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)) \
        if want_state else None
    y = None
    if g_in is not None:
        y = out["y"] if out else torch.empty((T, H, dv), dtype=torch.bfloat16, device=dev)
    args = make_prefill_args(q, k, v, z, beta, A, cu_seqlens, cu_host, o, S0=S0, S_T=S_T,
                             g_in=g_in, norm_w=norm_w, y=y, g_min=g_min, scale=scale,
                             qk_l2norm=qk_l2norm, norm_eps=norm_eps, gate=gate)
    S_snap = None
    if snap_interval:
        rows = snapshot_count(cu_host.tolist(), snap_interval)
        S_snap = torch.empty((max(rows, 1), H, dk, dv), dtype=torch.float32, device=dev)
        args.snap_interval = int(snap_interval)
        args.S_snap = S_snap.data_ptr()
        S_snap = S_snap[:rows]
    if not recurrent:
        need = prefill_workspace_size(args)
        if need > 0:
            # a caller's workspace is used as given: its size picks the schedule
            # (>= need: chunk-parallel; >= PREFILL_MIN_WORKSPACE: single pass);
            # "cache" reuses one buffer per device, grown on demand
            if isinstance(workspace, str) and workspace == "cache":
                key = (dev.type, dev.index)
                ws = _WS_CACHE.get(key)
                if ws is None or ws.numel() < need:
                    _WS_CACHE[key] = ws = torch.empty(need, dtype=torch.uint8, device=dev)
                workspace = ws
            elif workspace is None:
                workspace = torch.empty(need, dtype=torch.uint8, device=dev)
            args.workspace = workspace.data_ptr()
            args.workspace_bytes = workspace.numel() * workspace.element_size()
    prefill_raw(args, stream=stream, recurrent=recurrent)
    if snap_interval:
        return o, S_T, y, S_snap
    return o, S_T, y


SCAN_ZERO_V = 1   # kda_prefill_scan flag: evaluate with v = 0


class Records:
    """Chunk records of one set of prefill inputs (``kda_prefill_records``),
    kept with their inputs and workspace so that several ``prefill_scan``
    calls can run the state recurrence over them from different S0."""

    def __init__(self, args, keep, workspace, shape):
        self.args, self.keep, self.workspace, self.shape = args, keep, workspace, shape


def prefill_records(q, k, v, z, beta, A, cu_seqlens=None, g_min=-5.0, qk_l2norm=True, gate="bounded",
                    stream=None) -> Records:
    """Plan + prep of the chunk-parallel prefill through ``kda_prefill_records``."""
    T, H, dk = q.shape
    dev = q.device
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=dev)
    cu_host = cu_seqlens.to("cpu")
    args = make_prefill_args(q, k, v, z, beta, A, cu_seqlens, cu_host, None, g_min=g_min,
                             qk_l2norm=qk_l2norm, gate=gate)
    need = prefill_workspace_size(args)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    args.workspace, args.workspace_bytes = ws.data_ptr(), ws.numel()
    _check(load_library().kda_prefill_records(ctypes.byref(args), _stream(stream)), "kda_prefill_records")
    return Records(args, (q, k, v, z, beta, A, cu_seqlens, cu_host), ws, (T, H, dk, v.shape[2], cu_host.numel() - 1))


def prefill_scan(rec: Records, S0=None, g_in=None, norm_w=None, scale=1.0, norm_eps=1e-6, want_o=True,
                 want_state=True, zero_v=False, stream=None):
    """The state recurrence over ``rec`` through ``kda_prefill_scan``: returns
    (o, S_T, y) exactly as ``prefill`` would for the same inputs and S0
    (with v taken as zero when ``zero_v``)."""
    T, H, dk, dv, N = rec.shape
    dev = rec.workspace.device
    q = rec.keep[0]
    args = PrefillArgs.from_buffer_copy(rec.args)
    o = torch.empty((T, H, dv), dtype=q.dtype, device=dev) if want_o else None
    S_T = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev) if want_state else None
    y = torch.empty((T, H, dv), dtype=torch.bfloat16, device=dev) if g_in is not None else None
    for name, t in (("o", o), ("S0", S0), ("S_T", S_T), ("g_in", g_in), ("norm_w", norm_w), ("y", y)):
        setattr(args, name, t.data_ptr() if t is not None else None)
    args.scale, args.norm_eps = float(scale), float(norm_eps)
    _check(load_library().kda_prefill_scan(ctypes.byref(args), SCAN_ZERO_V if zero_v else 0, _stream(stream)),
           "kda_prefill_scan")
    return o, S_T, y


def make_decode_args(q, k, v, z, beta, A, state, o=None, y=None, g_in=None, norm_w=None,
                     slots=None, g_min=-5.0, scale=1.0, qk_l2norm=True, norm_eps=1e-6,
                     gate="bounded") -> DecodeArgs:
    N, H, dk = q.shape
    a = DecodeArgs()
    a.N, a.H, a.dk, a.dv = int(N), int(H), int(dk), int(v.shape[2])
    a.num_slots = int(state.shape[0])
    for name, t in (("q", q), ("k", k), ("v", v), ("z", z), ("beta", beta), ("A", A),
                    ("state", state), ("slots", slots), ("o", o), ("g_in", g_in),
                    ("norm_w", norm_w), ("y", y)):
        setattr(a, name, t.data_ptr() if t is not None else None)
    a.g_min, a.scale, a.qk_l2norm, a.norm_eps = float(g_min), float(scale), int(bool(qk_l2norm)), float(norm_eps)
    a.gate_mode = GATES[gate]
    return a


def decode_step_raw(args: DecodeArgs, stream=None):
    _check(load_library().kda_decode_step(ctypes.byref(args), _stream(stream)), "kda_decode_step")


def decode_step(q, k, v, z, beta, A, state, g_in=None, norm_w=None, slots=None, want_o=True,
                g_min=-5.0, scale=1.0, qk_l2norm=True, norm_eps=1e-6, stream=None, gate="bounded"):
    """One decode step through ``kda_decode_step``; ``state`` is updated in place.

    Returns (o or None, y or None).
    """
    N, H, _ = q.shape
    dv = v.shape[2]
    o = torch.empty((N, H, dv), dtype=torch.bfloat16, device=q.device) if want_o else None
    y = torch.empty((N, H, dv), dtype=torch.bfloat16, device=q.device) if g_in is not None else None
    args = make_decode_args(q, k, v, z, beta, A, state, o=o, y=y, g_in=g_in, norm_w=norm_w,
                            slots=slots, g_min=g_min, scale=scale, qk_l2norm=qk_l2norm,
                            norm_eps=norm_eps, gate=gate)
    decode_step_raw(args, stream)
    return o, y


def make_short_conv_args(x, weight, y, cu_seqlens, cu_seqlens_host, bias=None, state_in=None,
                         state_out=None, activation=True) -> ShortConvArgs:
    a = ShortConvArgs()
    a.num_seqs = int(cu_seqlens_host.numel() - 1)
    a.T_total, a.channels = int(x.shape[0]), int(x.shape[1])
    a.width = int(weight.shape[1])
    a.dtype = _dtype_code(x)
    a.cu_seqlens, a.cu_seqlens_host = cu_seqlens.data_ptr(), cu_seqlens_host.data_ptr()
    for name, t in (("x", x), ("weight", weight), ("bias", bias), ("state_in", state_in),
                    ("state_out", state_out), ("y", y)):
        setattr(a, name, t.data_ptr() if t is not None else None)
    a.activation = int(bool(activation))
    return a


def short_conv_raw(args: ShortConvArgs, stream=None):
    _check(load_library().kda_short_conv(ctypes.byref(args), _stream(stream)), "kda_short_conv")


def short_conv(x, weight, bias=None, cu_seqlens=None, state_in=None, want_state=True, activation=True,
               stream=None):
    """ShortConv + Swish prologue through ``kda_short_conv``.

    x: [T, C] (bf16 or f32); weight [C, W] f32; bias [C] or None; cu_seqlens int32
    [N+1] on the device (None = one sequence); state_in [N, W-1, C] f32 or None.
    Returns (y [T, C] in x's dtype, state_out [N, W-1, C] or None).
    """
    T, C = x.shape
    W = weight.shape[1]
    dev = x.device
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=dev)
    cu_host = cu_seqlens.to("cpu")
    N = cu_host.numel() - 1
    y = torch.empty_like(x)
    state_out = torch.empty((N, W - 1, C), dtype=torch.float32, device=dev) if (want_state and W > 1) else None
    args = make_short_conv_args(x, weight, y, cu_seqlens, cu_host, bias=bias, state_in=state_in,
                                state_out=state_out, activation=activation)
    short_conv_raw(args, stream)
    return y, state_out


def short_conv_step(x, weight, state, bias=None, slots=None, activation=True, stream=None):
    """One decode step of the prologue through ``kda_short_conv_step``; ``state``
    [S, W-1, C] is updated in place.  Returns y [N, C]."""
    N, C = x.shape
    a = ShortConvStepArgs()
    a.N, a.channels, a.width = int(N), int(C), int(weight.shape[1])
    a.num_slots = int(state.shape[0]) if state is not None else 0
    a.dtype = _dtype_code(x)
    y = torch.empty_like(x)
    for name, t in (("x", x), ("weight", weight), ("bias", bias), ("state", state), ("slots", slots), ("y", y)):
        setattr(a, name, t.data_ptr() if t is not None else None)
    a.activation = int(bool(activation))
    _check(load_library().kda_short_conv_step(ctypes.byref(a), _stream(stream)), "kda_short_conv_step")
    return y


def kcp_apply(M, X, add=None, stream=None):
    """X[h] <- M[h] X[h] + add[h] for every head, in place (``kda_kcp_apply``).
    M [H, d, d], X [H, d, n], add [H, d, n] or None; float32 on the device."""
    H, d, n = X.shape
    _check(load_library().kda_kcp_apply(_p(M), _p(X), _p(add), int(H), int(d), int(n), _stream(stream)),
           "kda_kcp_apply")
    return X


def gate_norm(o, g_in, norm_w=None, eps=1e-6, out=None, stream=None):
    """y = Sigmoid(g_in) * RMSNorm(o) through ``kda_gate_norm`` (rows over the last dim)."""
    dv = o.shape[-1]
    rows = o.numel() // dv
    y = out if out is not None else torch.empty_like(o)
    lib = load_library()
    _check(lib.kda_gate_norm(_p(o), _p(g_in), _p(norm_w), ctypes.c_float(eps), _p(y),
                             ctypes.c_long(rows), int(dv), _dtype_code(o), _stream(stream)),
           "kda_gate_norm")
    return y
