"""GB300 MoE expert block: thin Python binding of libmoe_gb300.so.

Every function here marshals torch tensors (device memory) and the current
CUDA stream into the C ABI of include/moe_expert.h and raises on a non-OK
status. All computation runs in the library's CUDA kernels; there is no
fallback: importing this package without the built library raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# MOE_GB300_DEBUG=1 loads the MOE_DEBUG build (device-side bounds checks of
# the row indices taken from row maps, reported as MOE_ERR_BOUNDS)
DEBUG = os.environ.get("MOE_GB300_DEBUG", "0") not in ("", "0")
# MOE_GB300_SANITIZE=1 loads the host-sanitizer build (AddressSanitizer and
# UndefinedBehaviorSanitizer on the host code; the process must preload their
# runtimes): it serves the host-side checks on a machine without a GPU
SANITIZE = os.environ.get("MOE_GB300_SANITIZE", "0") not in ("", "0")
LIB_PATH = os.path.join(_HERE, "libmoe_gb300_sanitize.so" if SANITIZE
                        else "libmoe_gb300_debug.so" if DEBUG else "libmoe_gb300.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python moe_expert_dispatch_gb300/build.py` "
        "(the expert block has no CPU or eager fallback)")

_lib = ctypes.CDLL(LIB_PATH)

MOE_OK = 0
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "expert id outside [0, E)",
          4: "workspace missing or too small", 5: "in-kernel wait timed out", 6: "CUDA error",
          7: "row index outside its buffer (debug build)"}
MOE_BF16, MOE_MXFP8 = 0, 1
TILE_M = 128

_vp, _i64, _i32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t


class moe_config(ctypes.Structure):
    _fields_ = [("ring_stages", ctypes.c_int), ("save_for_backward", ctypes.c_int),
                ("num_sms", ctypes.c_int), ("fuse_gather", ctypes.c_int),
                ("wait_limit_ns", ctypes.c_longlong),
                ("step_events", ctypes.POINTER(ctypes.c_void_p)),
                ("num_step_events", ctypes.c_int),
                ("mxfp8_tile_n", ctypes.c_int),
                ("cta_pairs", ctypes.c_int),
                ("mx_scales_pretiled", ctypes.c_int)]

STEP_EVENTS = 5       # forward: start, routing, fc1+SwiGLU, fc2, unpermute
BWD_STEP_EVENTS = 7   # backward: start, dO+dprobs, dH, dXp, dX, dW1, dW2
# MXFP8 backward: start, dO + quantise, dH, quantise dA, dXp, dX, quantise x and h, dW1, dW2
MX_BWD_STEP_EVENTS = 9


def _sig(name, res, *args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_sig("moe_config_init", None, ctypes.POINTER(moe_config))
_sig("moe_status_string", ctypes.c_char_p, _i32)
_sig("moe_get_error", _i32, _vp)
_sig("moe_num_sms", _i32)
_sig("moe_padded_rows", _i64, _i64, _i32, _i32)
_sig("moe_counts_workspace_size", _sz, _i64, _i32)
_sig("moe_counts", _i32, _vp, _i64, _i32, _vp, _vp, _vp, _sz, _vp)
_sig("moe_counts_static", _i32, _vp, _i64, _i32, _vp, _vp, _vp)
_sig("moe_route_topk_workspace_size", _sz, _i64, _i32, _i32)
_sig("moe_route_topk", _i32, _vp, _i64, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp)
_sig("moe_permute_workspace_size", _sz, _i64, _i32, _i32)
_sig("moe_permute", _i32, _vp, _i64, _i64, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp,
     _vp, _vp, _sz, _vp)
_sig("moe_unpermute", _i32, _vp, _vp, _vp, _i64, _i32, _i32, _vp, _vp)
_sig("moe_quantize_mxfp8", _i32, _vp, _i64, _i32, _vp, _vp, _vp)
_sig("moe_permute_quantize_mxfp8", _i32, _vp, _i64, _i32, _vp, _i32, _vp, _vp, _vp)
_sig("moe_workspace_size", _sz, _i64, _i32, _i32, _i32, _i32, ctypes.POINTER(moe_config), _i32)
_sig("moe_expert_forward", _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _i32, _vp,
     _vp, _sz, ctypes.POINTER(moe_config), _vp)
_sig("moe_expert_forward_from_logits", _i32, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32,
     _i32, _vp, _vp, _vp, _vp, _sz, ctypes.POINTER(moe_config), _vp)
_sig("moe_workspace_size_pipelined", _sz, _i64, _i32, _i32, _i32, _i32, _i32)
_sig("moe_expert_forward_pipelined", _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32,
     _i32, _vp, _i32, _vp, _sz, ctypes.POINTER(moe_config), _vp, _vp)
_sig("moe_expert_backward", _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32,
     _i32, _vp, _sz, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _sz, ctypes.POINTER(moe_config), _vp)
_sig("moe_workspace_size_mxfp8", _sz, _i64, _i32, _i32, _i32, _i32, ctypes.POINTER(moe_config))
_sig("moe_workspace_size_mxfp8_backward", _sz, _i64, _i32, _i32, _i32, _i32)
_sig("moe_quantize_mxfp8_t", _i32, _vp, _i64, _i32, _i32, _vp, _vp, _vp)
_sig("moe_quantize_mxfp8_dual", _i32, _vp, _i64, _i32, _i32, _vp, _vp, _vp, _vp, _vp)
_sig("moe_expert_backward_mxfp8", _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64,
     _i32, _i32, _i32, _i32, _vp, _sz, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _sz,
     ctypes.POINTER(moe_config), _vp)
_sig("moe_expert_forward_mxfp8", _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32,
     _i32, _i32, _i32, _vp, _vp, _sz, ctypes.POINTER(moe_config), _vp)
_sig("moe_tile_weight_scales_mxfp8", _i32, _vp, _vp, _vp, _i32, _i32, _i32,
     ctypes.POINTER(moe_config), _vp, _vp, _vp)


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, status)} (status {status})")
        self.status = status


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None, device=None):
    """The given stream, or the current stream of `device` (the device that
    the call's tensors live on); a given stream must belong to that device."""
    if stream is None:
        s = torch.cuda.current_stream(device)
    else:
        s = stream
        if device is not None and s.device != device:
            raise ValueError(f"stream is on {s.device}, the tensors on {device}")
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(t, name, dtype=None, min_numel=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs at least {min_numel}")


def _device(*named):
    """The one CUDA device of the (name, tensor) pairs given (None tensors
    skipped). Every kernel of a call runs on the device of its tensors, and
    a call whose tensors live on two devices is refused before anything is
    launched."""
    dev, first = None, None
    for name, t in named:
        if t is None:
            continue
        if dev is None:
            dev, first = t.device, name
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device} but {first} is on {dev}: "
                             "all tensors of a call must share one device")
    return dev


def config(ring_stages=0, save_for_backward=False, num_sms=0, fuse_gather=False,
           wait_limit_ns=0, step_events=None, mxfp8_tile_n=0, cta_pairs=0,
           mx_scales_pretiled=False) -> moe_config:
    """A moe_config; step_events: optional list of MOE_STEP_EVENTS torch.cuda.Event
    (already recorded once, so that their CUDA events exist)."""
    c = moe_config()
    _lib.moe_config_init(ctypes.byref(c))
    c.ring_stages = ring_stages
    c.save_for_backward = int(bool(save_for_backward))
    c.num_sms = num_sms
    c.fuse_gather = int(bool(fuse_gather))
    c.mxfp8_tile_n = mxfp8_tile_n
    c.cta_pairs = cta_pairs
    c.mx_scales_pretiled = int(bool(mx_scales_pretiled))
    if wait_limit_ns:
        c.wait_limit_ns = wait_limit_ns
    if step_events is not None:
        n = len(step_events)
        arr = (ctypes.c_void_p * n)(*[ev.cuda_event for ev in step_events])
        c._events_keepalive = arr
        c.step_events = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
        c.num_step_events = n
    return c


def moe_get_error(stream=None) -> int:
    """Synchronises the stream (default: the current device's current stream)
    and returns (and clears) the error status of the stream's device."""
    if stream is None:
        return _lib.moe_get_error(_stream(None))
    with torch.cuda.device(stream.device):
        return _lib.moe_get_error(_stream(stream))


def moe_num_sms() -> int:
    return _lib.moe_num_sms()


def moe_padded_rows(n_rows: int, E: int, row_align: int = TILE_M) -> int:
    return _lib.moe_padded_rows(n_rows, E, row_align)


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def moe_counts(expert_ids: torch.Tensor, num_experts: int, counts=None, offsets=None,
               workspace=None, stream=None):
    """(counts int32 [E], offsets int32 [E+1]) of the flattened ids."""
    _cuda(expert_ids, "expert_ids", torch.int32)
    _cuda(counts, "counts", torch.int32, num_experts)
    _cuda(offsets, "offsets", torch.int32, num_experts + 1)
    _cuda(workspace, "workspace")
    dev = _device(("expert_ids", expert_ids), ("counts", counts), ("offsets", offsets),
                  ("workspace", workspace))
    n = expert_ids.numel()
    with torch.cuda.device(dev):
        counts = (torch.empty(num_experts, dtype=torch.int32, device=dev)
                  if counts is None else counts)
        offsets = (torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
                   if offsets is None else offsets)
        need = _lib.moe_counts_workspace_size(n, num_experts)
        ws = _workspace(need, dev) if workspace is None else workspace
        _check(_lib.moe_counts(_p(expert_ids), n, num_experts, _p(counts), _p(offsets), _p(ws),
                               ws.numel(), _stream(stream, dev)), "moe_counts")
    return counts, offsets


def moe_route_topk(logits: torch.Tensor, k: int, expert_ids=None, probs=None, counts=None,
                   offsets=None, workspace=None, stream=None):
    """The top-k softmax gate fused with the counts: (expert_ids int32 [T, k],
    probs float32 [T, k], counts int32 [E], offsets int32 [E+1]) of float32
    router logits [T, E]."""
    _cuda(logits, "logits", torch.float32)
    T, E = logits.shape
    _cuda(expert_ids, "expert_ids", torch.int32, T * k)
    _cuda(probs, "probs", torch.float32, T * k)
    _cuda(counts, "counts", torch.int32, E)
    _cuda(offsets, "offsets", torch.int32, E + 1)
    _cuda(workspace, "workspace")
    dev = _device(("logits", logits), ("expert_ids", expert_ids), ("probs", probs),
                  ("counts", counts), ("offsets", offsets), ("workspace", workspace))
    with torch.cuda.device(dev):
        expert_ids = (torch.empty((T, k), dtype=torch.int32, device=dev)
                      if expert_ids is None else expert_ids)
        probs = torch.empty((T, k), dtype=torch.float32, device=dev) if probs is None else probs
        counts = torch.empty(E, dtype=torch.int32, device=dev) if counts is None else counts
        offsets = (torch.empty(E + 1, dtype=torch.int32, device=dev)
                   if offsets is None else offsets)
        need = _lib.moe_route_topk_workspace_size(T, k, E)
        ws = _workspace(need, dev) if workspace is None else workspace
        _check(_lib.moe_route_topk(_p(logits), T, E, k, _p(expert_ids), _p(probs), _p(counts),
                                   _p(offsets), _p(ws), ws.numel(), _stream(stream, dev)),
               "moe_route_topk")
    return expert_ids, probs, counts, offsets


def moe_counts_static(expert_ids: torch.Tensor, num_experts: int, counts=None, offsets=None,
                      stream=None):
    """moe_counts with the library's fixed scratch instead of a workspace: it
    allocates no device memory (the output tensors are created here only when
    the caller passes none). Calls that overlap on the GPU race on that scratch."""
    _cuda(expert_ids, "expert_ids", torch.int32)
    _cuda(counts, "counts", torch.int32, num_experts)
    _cuda(offsets, "offsets", torch.int32, num_experts + 1)
    dev = _device(("expert_ids", expert_ids), ("counts", counts), ("offsets", offsets))
    with torch.cuda.device(dev):        # the scratch used is the one of this device
        counts = (torch.empty(num_experts, dtype=torch.int32, device=dev)
                  if counts is None else counts)
        offsets = (torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
                   if offsets is None else offsets)
        _check(_lib.moe_counts_static(_p(expert_ids), expert_ids.numel(), num_experts,
                                      _p(counts), _p(offsets), _stream(stream, dev)),
               "moe_counts_static")
    return counts, offsets


def moe_permute(x: torch.Tensor, expert_ids: torch.Tensor, probs, num_experts: int,
                row_align: int = 1, stream=None):
    """Stable permute of token rows into expert-contiguous rows.

    Returns dict(x_perm, row_of, token_of, prob_of, offsets, counts). With
    row_align > 1 every expert segment starts at a multiple of row_align rows
    and the padding rows of x_perm/token_of/prob_of are left uninitialised.
    """
    _cuda(x, "x")
    _cuda(expert_ids, "expert_ids", torch.int32)
    _cuda(probs, "probs", torch.float32)
    T, k = expert_ids.shape
    dev = _device(("x", x), ("expert_ids", expert_ids), ("probs", probs))
    with torch.cuda.device(dev):
        return _moe_permute(x, expert_ids, probs, num_experts, row_align, stream, T, k, dev)


def _moe_permute(x, expert_ids, probs, num_experts, row_align, stream, T, k, dev):
    row_bytes = x[0].numel() * x.element_size() if T else x.element_size()
    cap = _lib.moe_padded_rows(T * k, num_experts, row_align)
    out = dict(
        x_perm=torch.empty((cap,) + tuple(x.shape[1:]), dtype=x.dtype, device=dev),
        row_of=torch.empty((T, k), dtype=torch.int32, device=dev),
        token_of=torch.empty(cap, dtype=torch.int32, device=dev),
        prob_of=torch.empty(cap, dtype=torch.float32, device=dev),
        offsets=torch.empty(num_experts + 1, dtype=torch.int32, device=dev),
        counts=torch.empty(num_experts, dtype=torch.int32, device=dev),
    )
    ws = _workspace(_lib.moe_permute_workspace_size(T, k, num_experts), dev)
    _check(_lib.moe_permute(_p(x), T, row_bytes, _p(expert_ids), _p(probs), k, num_experts,
                            row_align, _p(out["x_perm"]), _p(out["row_of"]), _p(out["token_of"]),
                            _p(out["prob_of"]), _p(out["offsets"]), _p(out["counts"]), _p(ws),
                            ws.numel(), _stream(stream, dev)), "moe_permute")
    return out


def moe_unpermute(o_perm: torch.Tensor, row_of: torch.Tensor, probs=None, y=None, stream=None):
    """y[t] = bf16(sum_j probs[t, j] * o_perm[row_of[t, j]])."""
    _cuda(o_perm, "o_perm", torch.bfloat16)
    _cuda(row_of, "row_of", torch.int32)
    T, k = row_of.shape
    H = o_perm.shape[-1]
    _cuda(probs, "probs", torch.float32, T * k)
    _cuda(y, "y", torch.bfloat16, T * H)
    dev = _device(("o_perm", o_perm), ("row_of", row_of), ("probs", probs), ("y", y))
    with torch.cuda.device(dev):
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if y is None else y
        _check(_lib.moe_unpermute(_p(o_perm), _p(row_of), _p(probs), T, k, H, _p(y),
                                  _stream(stream, dev)), "moe_unpermute")
    return y


def moe_quantize_mxfp8(a: torch.Tensor, stream=None, out=None):
    """(codes uint8 [..., K], scales uint8 [..., K/32]) of a bf16 tensor along
    its last axis, written into out=(codes, scales) when given."""
    _cuda(a, "a", torch.bfloat16)
    K = a.shape[-1]
    rows = a.numel() // K if K else 0
    if out is None:
        q = torch.empty(a.shape, dtype=torch.uint8, device=a.device)
        s = torch.empty(a.shape[:-1] + (K // 32,), dtype=torch.uint8, device=a.device)
    else:
        q, s = out
        _cuda(q, "q", torch.uint8, a.numel())
        _cuda(s, "scales", torch.uint8, a.numel() // 32)
    dev = _device(("a", a), ("q", q), ("scales", s))
    with torch.cuda.device(dev):
        _check(_lib.moe_quantize_mxfp8(_p(a), rows, K, _p(q), _p(s), _stream(stream, dev)),
               "moe_quantize_mxfp8")
    return q, s


def moe_permute_quantize_mxfp8(x: torch.Tensor, row_of: torch.Tensor, n_rows: int | None = None,
                               stream=None, out=None):
    """The MXFP8 dispatch of bf16 x [T, H]: (codes uint8 [n_rows, H] holding
    token t's codes at every row_of[t, j] >= 0, scales uint8 [T, H/32] in
    token order), written into out=(codes, scales) when given. n_rows
    defaults to T * k; rows that row_of does not name stay zero."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(row_of, "row_of", torch.int32)
    T, H = x.shape
    k = row_of.shape[1]
    if out is None:
        rows = T * k if n_rows is None else n_rows
        q = torch.zeros((rows, H), dtype=torch.uint8, device=x.device)
        s = torch.empty((T, H // 32), dtype=torch.uint8, device=x.device)
    else:
        q, s = out
        _cuda(q, "codes", torch.uint8)
        _cuda(s, "scales", torch.uint8, T * H // 32)
    dev = _device(("x", x), ("row_of", row_of), ("codes", q), ("scales", s))
    with torch.cuda.device(dev):
        _check(_lib.moe_permute_quantize_mxfp8(_p(x), T, H, _p(row_of), k, _p(q), _p(s),
                                               _stream(stream, dev)),
               "moe_permute_quantize_mxfp8")
    return q, s


def moe_quantize_mxfp8_t(a: torch.Tensor, stream=None, out=None):
    """MXFP8 along the rows of each matrix of a bf16 [batch, rows, cols] (or
    [rows, cols]) tensor: (codes uint8 [batch, cols, rows], scales uint8
    [batch, cols, rows/32]), written into out=(codes, scales) when given."""
    _cuda(a, "a", torch.bfloat16)
    squeeze = a.dim() == 2
    a3 = a.unsqueeze(0) if squeeze else a
    B, rows, cols = a3.shape
    if out is None:
        q = torch.empty((B, cols, rows), dtype=torch.uint8, device=a.device)
        s = torch.empty((B, cols, rows // 32), dtype=torch.uint8, device=a.device)
    else:
        q, s = out
        _cuda(q, "q", torch.uint8, a.numel())
        _cuda(s, "scales", torch.uint8, a.numel() // 32)
        if squeeze:
            q, s = q.unsqueeze(0), s.unsqueeze(0)
    dev = _device(("a", a), ("q", q), ("scales", s))
    with torch.cuda.device(dev):
        _check(_lib.moe_quantize_mxfp8_t(_p(a3), B, rows, cols, _p(q), _p(s),
                                         _stream(stream, dev)), "moe_quantize_mxfp8_t")
    return (q[0], s[0]) if squeeze else (q, s)


def moe_quantize_mxfp8_dual(a: torch.Tensor, stream=None, out=None):
    """Both orientations of a bf16 [batch, rows, cols] tensor from one read:
    (q [batch, rows, cols], s [batch, rows, cols/32]) as moe_quantize_mxfp8 and
    (qt [batch, cols, rows], st [batch, cols, rows/32]) as moe_quantize_mxfp8_t,
    written into out=(q, s, qt, st) when given."""
    _cuda(a, "a", torch.bfloat16)
    B, rows, cols = a.shape
    if out is None:
        out = (torch.empty((B, rows, cols), dtype=torch.uint8, device=a.device),
               torch.empty((B, rows, cols // 32), dtype=torch.uint8, device=a.device),
               torch.empty((B, cols, rows), dtype=torch.uint8, device=a.device),
               torch.empty((B, cols, rows // 32), dtype=torch.uint8, device=a.device))
    for t, n in zip(out, (a.numel(), a.numel() // 32, a.numel(), a.numel() // 32)):
        _cuda(t, "out", torch.uint8, n)
    dev = _device(("a", a), *(("out", t) for t in out))
    with torch.cuda.device(dev):
        _check(_lib.moe_quantize_mxfp8_dual(_p(a), B, rows, cols, *(_p(t) for t in out),
                                            _stream(stream, dev)), "moe_quantize_mxfp8_dual")
    return out


def moe_workspace_size(T, H, F, E, k, cfg: moe_config | None = None, for_backward=False) -> int:
    c = cfg if cfg is not None else config()
    return _lib.moe_workspace_size(T, H, F, E, k, ctypes.byref(c), int(for_backward))


def moe_expert_forward(x, w_gate, w_up, w_down, expert_ids, probs, y=None, workspace=None,
                       cfg: moe_config | None = None, stream=None):
    """y = the MoE expert block (counts, permute, fc1+SwiGLU, fc2, unpermute).

    Returns (y, workspace); with cfg.save_for_backward the workspace holds
    what moe_expert_backward needs."""
    for t, n in ((x, "x"), (w_gate, "w_gate"), (w_up, "w_up"), (w_down, "w_down")):
        _cuda(t, n, torch.bfloat16)
    _cuda(expert_ids, "expert_ids", torch.int32)
    _cuda(probs, "probs", torch.float32)
    T, H = x.shape
    E, _, F = w_gate.shape
    k = expert_ids.shape[1]
    _cuda(y, "y", torch.bfloat16, T * H)
    _cuda(workspace, "workspace")
    dev = _device(("x", x), ("w_gate", w_gate), ("w_up", w_up), ("w_down", w_down),
                  ("expert_ids", expert_ids), ("probs", probs), ("y", y),
                  ("workspace", workspace))
    c = cfg if cfg is not None else config()
    need = _lib.moe_workspace_size(T, H, F, E, k, ctypes.byref(c), 0)
    if need == 0 and T > 0:
        raise MoeError(1, "moe_workspace_size")
    with torch.cuda.device(dev):
        ws = _workspace(need, dev) if workspace is None else workspace
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if y is None else y
        _check(_lib.moe_expert_forward(_p(x), _p(w_gate), _p(w_up), _p(w_down), _p(expert_ids),
                                       _p(probs), T, H, F, E, k, _p(y), _p(ws), ws.numel(),
                                       ctypes.byref(c), _stream(stream, dev)),
               "moe_expert_forward")
    return y, ws


def moe_expert_forward_from_logits(x, w_gate, w_up, w_down, router_logits, k, y=None,
                                   expert_ids=None, probs=None, workspace=None,
                                   cfg: moe_config | None = None, stream=None):
    """moe_expert_forward with the fused gate in front: returns
    (y, expert_ids, probs, workspace), the routing as moe_route_topk gives it."""
    for t, n in ((x, "x"), (w_gate, "w_gate"), (w_up, "w_up"), (w_down, "w_down")):
        _cuda(t, n, torch.bfloat16)
    _cuda(router_logits, "router_logits", torch.float32)
    T, H = x.shape
    E, _, F = w_gate.shape
    _cuda(y, "y", torch.bfloat16, T * H)
    _cuda(expert_ids, "expert_ids", torch.int32, T * k)
    _cuda(probs, "probs", torch.float32, T * k)
    _cuda(workspace, "workspace")
    dev = _device(("x", x), ("w_gate", w_gate), ("w_up", w_up), ("w_down", w_down),
                  ("router_logits", router_logits), ("y", y), ("expert_ids", expert_ids),
                  ("probs", probs), ("workspace", workspace))
    c = cfg if cfg is not None else config()
    need = _lib.moe_workspace_size(T, H, F, E, k, ctypes.byref(c), 0)
    if need == 0 and T > 0:
        raise MoeError(1, "moe_workspace_size")
    with torch.cuda.device(dev):
        ws = _workspace(need, dev) if workspace is None else workspace
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if y is None else y
        expert_ids = (torch.empty((T, k), dtype=torch.int32, device=dev)
                      if expert_ids is None else expert_ids)
        probs = torch.empty((T, k), dtype=torch.float32, device=dev) if probs is None else probs
        _check(_lib.moe_expert_forward_from_logits(_p(x), _p(w_gate), _p(w_up), _p(w_down),
                                                   _p(router_logits), T, H, F, E, k,
                                                   _p(expert_ids), _p(probs), _p(y), _p(ws),
                                                   ws.numel(), ctypes.byref(c),
                                                   _stream(stream, dev)),
               "moe_expert_forward_from_logits")
    return y, expert_ids, probs, ws


_aux_streams = {}


def moe_expert_forward_pipelined(x, w_gate, w_up, w_down, expert_ids, probs, n_chunks, y=None,
                                 workspace=None, cfg: moe_config | None = None, stream=None,
                                 aux_stream=None):
    """moe_expert_forward over n_chunks token chunks, the routing of the next
    chunk and the combine of the last overlapping the GEMMs on a second
    stream (one cached per device unless aux_stream is given). Returns
    (y, workspace)."""
    for t, n in ((x, "x"), (w_gate, "w_gate"), (w_up, "w_up"), (w_down, "w_down")):
        _cuda(t, n, torch.bfloat16)
    _cuda(expert_ids, "expert_ids", torch.int32)
    _cuda(probs, "probs", torch.float32)
    T, H = x.shape
    E, _, F = w_gate.shape
    k = expert_ids.shape[1]
    _cuda(y, "y", torch.bfloat16, T * H)
    _cuda(workspace, "workspace")
    dev = _device(("x", x), ("w_gate", w_gate), ("w_up", w_up), ("w_down", w_down),
                  ("expert_ids", expert_ids), ("probs", probs), ("y", y),
                  ("workspace", workspace))
    c = cfg if cfg is not None else config()
    need = _lib.moe_workspace_size_pipelined(T, H, F, E, k, n_chunks)
    if need == 0 and T > 0:
        raise MoeError(1, "moe_workspace_size_pipelined")
    with torch.cuda.device(dev):
        ws = _workspace(need, dev) if workspace is None else workspace
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if y is None else y
        if aux_stream is None:
            aux_stream = _aux_streams.get(dev)
            if aux_stream is None:
                aux_stream = _aux_streams[dev] = torch.cuda.Stream(device=dev)
        _check(_lib.moe_expert_forward_pipelined(_p(x), _p(w_gate), _p(w_up), _p(w_down),
                                                 _p(expert_ids), _p(probs), T, H, F, E, k, _p(y),
                                                 n_chunks, _p(ws), ws.numel(), ctypes.byref(c),
                                                 _stream(stream, dev), _stream(aux_stream, dev)),
               "moe_expert_forward_pipelined")
    return y, ws


def moe_expert_backward(dy, x, w_gate, w_up, w_down, expert_ids, probs, fwd_workspace,
                        dx=None, dw_gate=None, dw_up=None, dw_down=None, dprobs=None,
                        accumulate_dw=False, workspace=None, cfg: moe_config | None = None,
                        stream=None):
    """Gradients (dx, dw_gate, dw_up, dw_down, dprobs) of moe_expert_forward."""
    for t, n in ((dy, "dy"), (x, "x"), (w_gate, "w_gate"), (w_up, "w_up"), (w_down, "w_down")):
        _cuda(t, n, torch.bfloat16)
    _cuda(expert_ids, "expert_ids", torch.int32)
    _cuda(probs, "probs", torch.float32)
    _cuda(fwd_workspace, "fwd_workspace")
    T, H = x.shape
    E, _, F = w_gate.shape
    k = expert_ids.shape[1]
    _cuda(dx, "dx", torch.bfloat16, T * H)
    for t, n in ((dw_gate, "dw_gate"), (dw_up, "dw_up"), (dw_down, "dw_down")):
        _cuda(t, n, torch.float32, E * H * F)
    _cuda(dprobs, "dprobs", torch.float32, T * k)
    _cuda(workspace, "workspace")
    dev = _device(("dy", dy), ("x", x), ("w_gate", w_gate), ("w_up", w_up), ("w_down", w_down),
                  ("expert_ids", expert_ids), ("probs", probs), ("fwd_workspace", fwd_workspace),
                  ("dx", dx), ("dw_gate", dw_gate), ("dw_up", dw_up), ("dw_down", dw_down),
                  ("dprobs", dprobs), ("workspace", workspace))
    c = cfg if cfg is not None else config(save_for_backward=True)
    with torch.cuda.device(dev):
        dx = torch.empty_like(x) if dx is None else dx
        f32 = dict(dtype=torch.float32, device=dev)
        dw_gate = torch.empty((E, H, F), **f32) if dw_gate is None else dw_gate
        dw_up = torch.empty((E, H, F), **f32) if dw_up is None else dw_up
        dw_down = torch.empty((E, F, H), **f32) if dw_down is None else dw_down
        dprobs = torch.empty((T, k), **f32) if dprobs is None else dprobs
        need = _lib.moe_workspace_size(T, H, F, E, k, ctypes.byref(c), 1)
        ws = _workspace(need, dev) if workspace is None else workspace
        _check(_lib.moe_expert_backward(_p(dy), _p(x), _p(w_gate), _p(w_up), _p(w_down),
                                        _p(expert_ids), _p(probs), T, H, F, E, k,
                                        _p(fwd_workspace), fwd_workspace.numel(), _p(dx),
                                        _p(dw_gate), _p(dw_up), _p(dw_down), _p(dprobs),
                                        int(bool(accumulate_dw)), _p(ws), ws.numel(),
                                        ctypes.byref(c), _stream(stream, dev)),
               "moe_expert_backward")
    return dict(dx=dx, dw_gate=dw_gate, dw_up=dw_up, dw_down=dw_down, dprobs=dprobs)


def moe_workspace_size_mxfp8(T, H, F, E, k, cfg: moe_config | None = None) -> int:
    c = cfg if cfg is not None else config()
    return _lib.moe_workspace_size_mxfp8(T, H, F, E, k, ctypes.byref(c))


def moe_workspace_size_mxfp8_backward(T, H, F, E, k) -> int:
    return _lib.moe_workspace_size_mxfp8_backward(T, H, F, E, k)


def moe_tile_weight_scales_mxfp8(wg_s, wu_s, wd_s, cfg: moe_config | None = None, stream=None,
                                 out=None):
    """The weights' scales laid out once for the MXFP8 forward's block-scaled
    MMAs: (wgu_tiled, wd_tiled), to pass as wg_s and wd_s to
    moe_expert_forward_mxfp8 with config(mx_scales_pretiled=True) and the same
    mxfp8_tile_n. wg_s, wu_s [E, F, H/32], wd_s [E, H, F/32] as
    moe_quantize_mxfp8 writes them."""
    for t, n in ((wg_s, "wg_s"), (wu_s, "wu_s"), (wd_s, "wd_s")):
        _cuda(t, n, torch.uint8)
    E, F, H32 = wg_s.shape
    H = 32 * H32
    if tuple(wu_s.shape) != (E, F, H32) or tuple(wd_s.shape) != (E, H, F // 32):
        raise ValueError("wg_s, wu_s [E, F, H/32] and wd_s [E, H, F/32] expected")
    if out is None:
        wgu = torch.empty(E * 2 * F * H32, dtype=torch.uint8, device=wg_s.device)
        wdt = torch.empty(E * H * (F // 32), dtype=torch.uint8, device=wg_s.device)
    else:
        wgu, wdt = out
        _cuda(wgu, "wgu_tiled", torch.uint8, E * 2 * F * H32)
        _cuda(wdt, "wd_tiled", torch.uint8, E * H * (F // 32))
    dev = _device(("wg_s", wg_s), ("wu_s", wu_s), ("wd_s", wd_s), ("wgu_tiled", wgu),
                  ("wd_tiled", wdt))
    c = cfg if cfg is not None else config()
    with torch.cuda.device(dev):
        _check(_lib.moe_tile_weight_scales_mxfp8(_p(wg_s), _p(wu_s), _p(wd_s), H, F, E,
                                                 ctypes.byref(c), _p(wgu), _p(wdt),
                                                 _stream(stream, dev)),
               "moe_tile_weight_scales_mxfp8")
    return wgu, wdt


def moe_expert_forward_mxfp8(x, wg_q, wg_s, wu_q, wu_s, wd_q, wd_s, expert_ids, probs, y=None,
                             workspace=None, cfg: moe_config | None = None, stream=None):
    """The block with MXFP8 operands (x quantised on the fly; weights pre-quantised,
    K-contiguous: wg/wu [E, F, H], wd [E, H, F], scales [..., K/32]). With
    cfg.mx_scales_pretiled, wg_s and wd_s are moe_tile_weight_scales_mxfp8's
    outputs and wu_s may be None."""
    _cuda(x, "x", torch.bfloat16)
    for t, n in ((wg_q, "wg_q"), (wg_s, "wg_s"), (wu_q, "wu_q"), (wu_s, "wu_s"), (wd_q, "wd_q"),
                 (wd_s, "wd_s")):
        _cuda(t, n, torch.uint8)
    _cuda(expert_ids, "expert_ids", torch.int32)
    _cuda(probs, "probs", torch.float32)
    T, H = x.shape
    E, F, _ = wg_q.shape
    k = expert_ids.shape[1]
    _cuda(y, "y", torch.bfloat16, T * H)
    _cuda(workspace, "workspace")
    dev = _device(("x", x), ("wg_q", wg_q), ("wg_s", wg_s), ("wu_q", wu_q), ("wu_s", wu_s),
                  ("wd_q", wd_q), ("wd_s", wd_s), ("expert_ids", expert_ids), ("probs", probs),
                  ("y", y), ("workspace", workspace))
    c = cfg if cfg is not None else config()
    need = _lib.moe_workspace_size_mxfp8(T, H, F, E, k, ctypes.byref(c))
    with torch.cuda.device(dev):
        ws = _workspace(need, dev) if workspace is None else workspace
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if y is None else y
        _check(_lib.moe_expert_forward_mxfp8(_p(x), _p(wg_q), _p(wg_s), _p(wu_q), _p(wu_s),
                                             _p(wd_q), _p(wd_s), _p(expert_ids), _p(probs), T, H,
                                             F, E, k, _p(y), _p(ws), ws.numel(), ctypes.byref(c),
                                             _stream(stream, dev)), "moe_expert_forward_mxfp8")
    return y, ws


def moe_expert_backward_mxfp8(dy, x, w1g_q, w1g_s, w1u_q, w1u_s, w2_q, w2_s, expert_ids, probs,
                              fwd_workspace, dx=None, dw_gate_t=None, dw_up_t=None,
                              dw_down_t=None, dprobs=None, accumulate_dw=False, workspace=None,
                              cfg: moe_config | None = None, stream=None):
    """Gradients of moe_expert_forward_mxfp8 (run with save_for_backward):
    dict(dx, dw_gate_t [E, F, H], dw_up_t [E, F, H], dw_down_t [E, H, F],
    dprobs). The weights come in the backward orientation of
    moe_quantize_mxfp8_t: w1g/w1u [E, H, F], w2 [E, F, H]."""
    for t, n in ((dy, "dy"), (x, "x")):
        _cuda(t, n, torch.bfloat16)
    for t, n in ((w1g_q, "w1g_q"), (w1g_s, "w1g_s"), (w1u_q, "w1u_q"), (w1u_s, "w1u_s"),
                 (w2_q, "w2_q"), (w2_s, "w2_s")):
        _cuda(t, n, torch.uint8)
    _cuda(expert_ids, "expert_ids", torch.int32)
    _cuda(probs, "probs", torch.float32)
    _cuda(fwd_workspace, "fwd_workspace")
    T, H = x.shape
    E, _, F = w1g_q.shape
    k = expert_ids.shape[1]
    _cuda(dx, "dx", torch.bfloat16, T * H)
    for t, n in ((dw_gate_t, "dw_gate_t"), (dw_up_t, "dw_up_t"), (dw_down_t, "dw_down_t")):
        _cuda(t, n, torch.float32, E * H * F)
    _cuda(dprobs, "dprobs", torch.float32, T * k)
    _cuda(workspace, "workspace")
    dev = _device(("dy", dy), ("x", x), ("w1g_q", w1g_q), ("w1g_s", w1g_s), ("w1u_q", w1u_q),
                  ("w1u_s", w1u_s), ("w2_q", w2_q), ("w2_s", w2_s), ("expert_ids", expert_ids),
                  ("probs", probs), ("fwd_workspace", fwd_workspace), ("dx", dx),
                  ("dw_gate_t", dw_gate_t), ("dw_up_t", dw_up_t), ("dw_down_t", dw_down_t),
                  ("dprobs", dprobs), ("workspace", workspace))
    c = cfg if cfg is not None else config(save_for_backward=True)
    with torch.cuda.device(dev):
        dx = torch.empty_like(x) if dx is None else dx
        f32 = dict(dtype=torch.float32, device=dev)
        dw_gate_t = torch.empty((E, F, H), **f32) if dw_gate_t is None else dw_gate_t
        dw_up_t = torch.empty((E, F, H), **f32) if dw_up_t is None else dw_up_t
        dw_down_t = torch.empty((E, H, F), **f32) if dw_down_t is None else dw_down_t
        dprobs = torch.empty((T, k), **f32) if dprobs is None else dprobs
        need = _lib.moe_workspace_size_mxfp8_backward(T, H, F, E, k)
        ws = _workspace(need, dev) if workspace is None else workspace
        _check(_lib.moe_expert_backward_mxfp8(_p(dy), _p(x), _p(w1g_q), _p(w1g_s), _p(w1u_q),
                                              _p(w1u_s), _p(w2_q), _p(w2_s), _p(expert_ids),
                                              _p(probs), T, H, F, E, k, _p(fwd_workspace),
                                              fwd_workspace.numel(), _p(dx), _p(dw_gate_t),
                                              _p(dw_up_t), _p(dw_down_t), _p(dprobs),
                                              int(bool(accumulate_dw)), _p(ws), ws.numel(),
                                              ctypes.byref(c), _stream(stream, dev)),
               "moe_expert_backward_mxfp8")
    return dict(dx=dx, dw_gate_t=dw_gate_t, dw_up_t=dw_up_t, dw_down_t=dw_down_t, dprobs=dprobs)
