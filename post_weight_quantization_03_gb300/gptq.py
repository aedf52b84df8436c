"""Thin Python binding of ``libgptq.so`` (argument marshalling only).

The functions named like the C entry points (``gptq_hessian_accumulate``, ``gptq_prepare``,
``gptq_quantize_layer``, ...) take raw device pointers, sizes and a stream handle exactly as
the C ABI does.  The tensor helpers below them (``hessian``, ``prepare``, ``quantize``) only
allocate outputs/workspaces with torch, pass pointers, and raise on a non-OK status: every
step of the computation runs in the library's CUDA kernels.  There is no fallback: if the
library is missing or fails to load, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import re

from . import build_lib

GPTQ_OK = 0
STATUS_NAMES = {
    0: "GPTQ_OK", 1: "GPTQ_ERR_INVALID_ARG", 2: "GPTQ_ERR_NOT_PD", 3: "GPTQ_ERR_NONFINITE",
    4: "GPTQ_ERR_TIMEOUT", 5: "GPTQ_ERR_CUDA", 6: "GPTQ_ERR_UNSUPPORTED", 7: "GPTQ_ERR_WORKSPACE",
}
DTYPES = {"f16": 0, "bf16": 1, "f32": 2}

_c = ctypes
_SIGS = {
    "gptq_status_str": (_c.c_char_p, [_c.c_int]),
    "gptq_abi_version": (_c.c_int, []),
    "gptq_kernel_launches": (_c.c_ulonglong, []),
    "gptq_hessian_accumulate": (_c.c_int, [_c.c_void_p, _c.c_int, _c.c_int64, _c.c_int64,
                                           _c.c_int64, _c.c_void_p, _c.c_int, _c.c_void_p]),
    "gptq_hessian_host_workspace_bytes": (_c.c_size_t, [_c.c_int, _c.c_int64, _c.c_int64]),
    "gptq_hessian_accumulate_host": (_c.c_int, [_c.c_void_p, _c.c_int, _c.c_int64, _c.c_int64,
                                                _c.c_int64, _c.c_void_p, _c.c_int, _c.c_int64,
                                                _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    "gptq_prepare_workspace_bytes": (_c.c_size_t, [_c.c_int64]),
    "gptq_prepare": (_c.c_int, [_c.c_void_p, _c.c_int64, _c.c_float, _c.c_void_p, _c.c_void_p,
                                _c.c_void_p, _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    "gptq_quantize_workspace_bytes": (_c.c_size_t, [_c.c_int64, _c.c_int64, _c.c_int, _c.c_int]),
    "gptq_quantize_layer": (_c.c_int, [_c.c_void_p, _c.c_int, _c.c_int64, _c.c_int64,
                                       _c.c_int64, _c.c_void_p, _c.c_void_p, _c.c_int,
                                       _c.c_int, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                       _c.c_void_p, _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    "gptq_workspace_status": (_c.c_int, [_c.c_void_p, _c.c_void_p]),
    "gptq_recon_error_workspace_bytes": (_c.c_size_t, [_c.c_int, _c.c_int64, _c.c_int64,
                                                       _c.c_int64]),
    "gptq_recon_error": (_c.c_int, [_c.c_void_p, _c.c_int, _c.c_int64, _c.c_int64, _c.c_int64,
                                    _c.c_void_p, _c.c_int, _c.c_int64, _c.c_int64, _c.c_void_p,
                                    _c.c_int, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                    _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    "gptq_quantize_obq_workspace_bytes": (_c.c_size_t, [_c.c_int64, _c.c_int64]),
    "gptq_quantize_obq": (_c.c_int, [_c.c_void_p, _c.c_int, _c.c_int64, _c.c_int64, _c.c_int64,
                                     _c.c_void_p, _c.c_void_p, _c.c_int, _c.c_void_p,
                                     _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                     _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    "gptq_quantize_shared_workspace_bytes": (_c.c_size_t, [_c.c_int, _c.c_void_p, _c.c_int64,
                                                           _c.c_int, _c.c_int]),
    "gptq_quantize_layers_shared": (_c.c_int, [_c.c_int, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                               _c.c_void_p, _c.c_int64, _c.c_void_p,
                                               _c.c_void_p, _c.c_int, _c.c_int, _c.c_void_p,
                                               _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                               _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    "gptq_quantize_layer_noalloc": (_c.c_int, [_c.c_void_p, _c.c_int, _c.c_int64, _c.c_int64,
                                               _c.c_int64, _c.c_void_p, _c.c_void_p, _c.c_int,
                                               _c.c_int, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                               _c.c_void_p, _c.c_void_p]),
    "gptq_noalloc_status": (_c.c_int, [_c.c_void_p]),
    "gptq_debug_hessian_lost_stage": (_c.c_int, [_c.c_void_p, _c.c_int, _c.c_int64, _c.c_int64,
                                                 _c.c_int64, _c.c_void_p, _c.c_int64,
                                                 _c.c_uint64, _c.c_void_p, _c.c_void_p]),
}
NOALLOC_SCRATCH_BYTES = 32 << 20  # GPTQ_NOALLOC_SCRATCH_BYTES in include/gptq.h
OBQ_MAX_D_IN = 128                # GPTQ_OBQ_MAX_D_IN in include/gptq.h
MAX_SHARED_LAYERS = 64            # GPTQ_MAX_SHARED_LAYERS in include/gptq.h

_lib = None


class GptqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS_NAMES.get(self.status, self.status)}")


def library_path() -> str:
    return build_lib.LIB


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the library (once).  Raises if it is missing: build it with
    ``python -m post_weight_quantization_03_gb300.build_lib``."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or library_path()
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: the CUDA library must be built (build_lib.build())")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def declared_symbols(header: str | None = None):
    """Names of the functions ``include/gptq.h`` declares."""
    header = header or os.path.join(build_lib.INCLUDE, "gptq.h")
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gptq_[a-z_0-9]+)\s*\(", text)))


# ---------------------------------------------------------------------------------------
# C entry points, same names and arguments
# ---------------------------------------------------------------------------------------

def gptq_status_str(status):
    return load().gptq_status_str(status).decode()


def gptq_abi_version():
    return load().gptq_abi_version()


def gptq_kernel_launches():
    return load().gptq_kernel_launches()


def gptq_hessian_accumulate(X, xdtype, n_tok, d_in, ldx, H, accumulate, stream):
    return load().gptq_hessian_accumulate(X, xdtype, n_tok, d_in, ldx, H, accumulate, stream)


def gptq_hessian_host_workspace_bytes(xdtype, d_in, chunk_tok):
    return load().gptq_hessian_host_workspace_bytes(xdtype, d_in, chunk_tok)


def gptq_hessian_accumulate_host(X_host, xdtype, n_tok, d_in, ldx, H, accumulate, chunk_tok, ws,
                                 ws_bytes, stream):
    return load().gptq_hessian_accumulate_host(X_host, xdtype, n_tok, d_in, ldx, H, accumulate,
                                               chunk_tok, ws, ws_bytes, stream)


def gptq_prepare_workspace_bytes(d_in):
    return load().gptq_prepare_workspace_bytes(d_in)


def gptq_prepare(H, d_in, damp, U, dead_mask, n_dead, ws, ws_bytes, stream):
    return load().gptq_prepare(H, d_in, damp, U, dead_mask, n_dead, ws, ws_bytes, stream)


def gptq_quantize_workspace_bytes(d_out, d_in, bits, block):
    return load().gptq_quantize_workspace_bytes(d_out, d_in, bits, block)


def gptq_quantize_layer(W, wdtype, d_out, d_in, ldw, U, dead_mask, bits, block, qpacked,
                        scale, zero, W_hat, ws, ws_bytes, stream):
    return load().gptq_quantize_layer(W, wdtype, d_out, d_in, ldw, U, dead_mask, bits, block,
                                      qpacked, scale, zero, W_hat, ws, ws_bytes, stream)


def gptq_workspace_status(ws, stream):
    return load().gptq_workspace_status(ws, stream)


def gptq_recon_error_workspace_bytes(xdtype, d_out, d_in, n_tok):
    return load().gptq_recon_error_workspace_bytes(xdtype, d_out, d_in, n_tok)


def gptq_recon_error(X, xdtype, n_tok, d_in, ldx, W, wdtype, d_out, ldw, qpacked, bits, scale,
                     zero, err, ws, ws_bytes, stream):
    return load().gptq_recon_error(X, xdtype, n_tok, d_in, ldx, W, wdtype, d_out, ldw, qpacked,
                                   bits, scale, zero, err, ws, ws_bytes, stream)


def gptq_quantize_obq_workspace_bytes(d_out, d_in):
    return load().gptq_quantize_obq_workspace_bytes(d_out, d_in)


def gptq_quantize_obq(W, wdtype, d_out, d_in, ldw, U, dead_mask, bits, qpacked, scale, zero,
                      W_hat, order, ws, ws_bytes, stream):
    return load().gptq_quantize_obq(W, wdtype, d_out, d_in, ldw, U, dead_mask, bits, qpacked,
                                    scale, zero, W_hat, order, ws, ws_bytes, stream)


def gptq_quantize_shared_workspace_bytes(n_layers, d_out, d_in, bits, block):
    return load().gptq_quantize_shared_workspace_bytes(n_layers, d_out, d_in, bits, block)


def gptq_quantize_layers_shared(n_layers, W, wdtype, d_out, ldw, d_in, U, dead_mask, bits, block,
                                qpacked, scale, zero, W_hat, ws, ws_bytes, stream):
    return load().gptq_quantize_layers_shared(n_layers, W, wdtype, d_out, ldw, d_in, U,
                                              dead_mask, bits, block, qpacked, scale, zero,
                                              W_hat, ws, ws_bytes, stream)


def gptq_quantize_layer_noalloc(W, wdtype, d_out, d_in, ldw, U, dead_mask, bits, block,
                                qpacked, scale, zero, W_hat, stream):
    return load().gptq_quantize_layer_noalloc(W, wdtype, d_out, d_in, ldw, U, dead_mask, bits,
                                              block, qpacked, scale, zero, W_hat, stream)


def gptq_noalloc_status(stream):
    return load().gptq_noalloc_status(stream)


def gptq_debug_hessian_lost_stage(X, xdtype, n_tok, d_in, ldx, H, lost_stage, wait_ns, status_ws,
                                  stream):
    return load().gptq_debug_hessian_lost_stage(X, xdtype, n_tok, d_in, ldx, H, lost_stage,
                                                wait_ns, status_ws, stream)


# ---------------------------------------------------------------------------------------
# torch-tensor helpers (marshalling only)
# ---------------------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    m = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}
    if t.dtype not in m:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return m[t.dtype]


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status, where):
    if status != GPTQ_OK:
        raise GptqError(status, where)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def workspace(nbytes, device):
    """A 256-byte aligned byte workspace (torch allocations are 256-byte aligned)."""
    torch = _torch()
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


def hessian(X, H=None, accumulate=False, stream=None):
    """``H (+)= 2 X^T X`` for token-major X ``[n_tok, d_in]`` (row stride X.stride(0))."""
    torch = _torch()
    if X.dim() != 2 or X.stride(1) != 1:
        raise ValueError("X must be a row-major [n_tok, d_in] matrix")
    n, d = X.shape
    if H is None:
        H = torch.empty(d, d, dtype=torch.float32, device=X.device)
        accumulate = False
    _check(gptq_hessian_accumulate(_ptr(X), _dtype_code(X), n, d, X.stride(0), _ptr(H),
                                   1 if accumulate else 0, _stream(stream)),
           "gptq_hessian_accumulate")
    return H


def hessian_host(Xh, H=None, accumulate=False, chunk_tok=0, ws=None, device=None, stream=None):
    """``H (+)= 2 X^T X`` for a token-major HOST matrix ``Xh`` (CPU tensor, pinned for the
    copies to overlap), streamed to the device in chunks of ``chunk_tok`` tokens."""
    torch = _torch()
    if Xh.device.type != "cpu" or Xh.dim() != 2 or Xh.stride(1) != 1:
        raise ValueError("Xh must be a row-major [n_tok, d_in] CPU matrix")
    n, d = Xh.shape
    dev = torch.device(device) if device is not None else (
        H.device if H is not None else torch.device("cuda", torch.cuda.current_device()))
    if H is None:
        H = torch.empty(d, d, dtype=torch.float32, device=dev)
        accumulate = False
    need = gptq_hessian_host_workspace_bytes(_dtype_code(Xh), d, chunk_tok)
    if ws is None:
        ws = workspace(need, H.device)
    _check(gptq_hessian_accumulate_host(ctypes.c_void_p(Xh.data_ptr()), _dtype_code(Xh), n, d,
                                        Xh.stride(0), _ptr(H), 1 if accumulate else 0, chunk_tok,
                                        _ptr(ws), ws.numel(), _stream(stream)),
           "gptq_hessian_accumulate_host")
    return H


def prepare(H, damp=0.01, U=None, dead_mask=None, ws=None, stream=None):
    """Dead columns + damping + ``U`` with ``U^T U = H_damped^-1``.  CONSUMES ``H``.

    Returns ``(U, dead_mask, n_dead)``.
    """
    torch = _torch()
    d = H.shape[0]
    if H.dtype != torch.float32 or not H.is_contiguous() or H.shape != (d, d):
        raise ValueError("H must be a contiguous float32 [d, d] matrix")
    if U is None:
        U = torch.empty(d, d, dtype=torch.float32, device=H.device)
    if dead_mask is None:
        dead_mask = torch.empty(d, dtype=torch.uint8, device=H.device)
    nbytes = gptq_prepare_workspace_bytes(d)
    if ws is None:
        ws = workspace(nbytes, H.device)
    n_dead = ctypes.c_int32(0)
    _check(gptq_prepare(_ptr(H), d, float(damp), _ptr(U), _ptr(dead_mask),
                        ctypes.byref(n_dead), _ptr(ws), ws.numel(), _stream(stream)),
           "gptq_prepare")
    return U, dead_mask, n_dead.value


def packed_words(d_in, bits):
    return ((d_in + 31) // 32) * bits


def quantize(W, U, bits=4, block=128, dead_mask=None, want_w_hat=True, ws=None, stream=None,
             out=None):
    """The GPTQ sweep of one layer.  Returns ``(qpacked, scale, zero, W_hat or None)``."""
    torch = _torch()
    if W.dim() != 2 or W.stride(1) != 1:
        raise ValueError("W must be a row-major [d_out, d_in] matrix")
    m, d = W.shape
    dev = W.device
    if out is None:
        qpacked = torch.empty(m, packed_words(d, bits), dtype=torch.int32, device=dev)
        scale = torch.empty(m, dtype=torch.float32, device=dev)
        zero = torch.empty(m, dtype=torch.int32, device=dev)
        W_hat = torch.empty(m, d, dtype=torch.float32, device=dev) if want_w_hat else None
    else:
        qpacked, scale, zero, W_hat = out
    if ws is None:
        ws = workspace(gptq_quantize_workspace_bytes(m, d, bits, block), dev)
    _check(gptq_quantize_layer(_ptr(W), _dtype_code(W), m, d, W.stride(0), _ptr(U),
                               _ptr(dead_mask), bits, block, _ptr(qpacked), _ptr(scale),
                               _ptr(zero), _ptr(W_hat), _ptr(ws), ws.numel(), _stream(stream)),
           "gptq_quantize_layer")
    return qpacked, scale, zero, W_hat


def _ptr_array(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() if t is not None else None for t in ts])


def quantize_shared(Ws, U, bits=4, block=128, dead_mask=None, want_w_hat=False, ws=None,
                    stream=None):
    """The sweep of several layers sharing U (one stack of rows).  Returns one
    ``(qpacked, scale, zero, W_hat or None)`` tuple per layer."""
    torch = _torch()
    n = len(Ws)
    d = Ws[0].shape[1]
    for W in Ws:
        if W.dim() != 2 or W.stride(1) != 1 or W.shape[1] != d:
            raise ValueError("every W must be a row-major [d_out, d_in] matrix with one d_in")
    dev = Ws[0].device
    outs = []
    for W in Ws:
        m = W.shape[0]
        outs.append((torch.empty(m, packed_words(d, bits), dtype=torch.int32, device=dev),
                     torch.empty(m, dtype=torch.float32, device=dev),
                     torch.empty(m, dtype=torch.int32, device=dev),
                     torch.empty(m, d, dtype=torch.float32, device=dev) if want_w_hat else None))
    d_out = (ctypes.c_int64 * n)(*[W.shape[0] for W in Ws])
    if ws is None:
        ws = workspace(gptq_quantize_shared_workspace_bytes(n, d_out, d, bits, block), dev)
    _check(gptq_quantize_layers_shared(
        n, _ptr_array(Ws), (ctypes.c_int * n)(*[_dtype_code(W) for W in Ws]), d_out,
        (ctypes.c_int64 * n)(*[W.stride(0) for W in Ws]), d, _ptr(U), _ptr(dead_mask), bits,
        block, _ptr_array([o[0] for o in outs]), _ptr_array([o[1] for o in outs]),
        _ptr_array([o[2] for o in outs]),
        _ptr_array([o[3] for o in outs]) if want_w_hat else None, _ptr(ws), ws.numel(),
        _stream(stream)), "gptq_quantize_layers_shared")
    return outs


def quantize_block(groups, bits=(4,), block=128, damp=0.01, chunk_tok=None, overlap=True,
                   stage_events=None, consumers=2):
    """GPTQ over a block of layers grouped by their shared inputs.

    ``groups`` is a list of ``(X, [W, ...])``: X the token-major inputs of the group (on the
    device) and the weights of every layer that reads them.  Per group: H from X, one
    prepare, then one shared sweep of all its layers per bit width.  With ``overlap`` the
    Hessians are accumulated (in chunks of ``chunk_tok`` tokens, or in one call when None) on
    a producer stream, ahead of the prepares and sweeps, which run on ``consumers``
    higher-priority streams taken in turn by group (so one group's sweep can run beside the
    next group's prepare); every step is a call of this library.  Returns
    ``[{bits: [(qpacked, scale, zero, None) per layer]}, ...]`` and the dead-column counts,
    in group order."""
    torch = _torch()
    dev = groups[0][1][0].device
    caller = torch.cuda.current_stream(dev)
    lo, hi = torch.cuda.Stream.priority_range()
    cons_all = ([torch.cuda.Stream(dev, priority=hi) for _ in range(max(1, consumers))]
                if overlap else [caller])
    prod = torch.cuda.Stream(dev, priority=lo) if overlap else caller
    if overlap:
        prod.wait_stream(caller)
        for c in cons_all:
            c.wait_stream(caller)
    Hs, ready = [], []
    for X, _ in groups:
        d = X.shape[1]
        H = torch.empty(d, d, dtype=torch.float32, device=dev)
        if stage_events is not None:
            e0 = torch.cuda.Event(enable_timing=True)
            e0.record(prod)
        step = chunk_tok or max(X.shape[0], 1)
        for t0 in range(0, X.shape[0], step):
            hessian(X[t0:t0 + step], H, accumulate=t0 > 0, stream=prod)
        e = torch.cuda.Event(enable_timing=stage_events is not None)
        e.record(prod)
        if stage_events is not None:
            stage_events.append(("hessian", e0, e))
        Hs.append(H)
        ready.append(e)
    results, n_dead, keep = [], [], []
    for gi, ((X, Ws), H, e) in enumerate(zip(groups, Hs, ready)):
        cons = cons_all[gi % len(cons_all)]
        cons.wait_event(e)
        d = X.shape[1]
        e0 = torch.cuda.Event(enable_timing=True)
        e0.record(cons)
        # every buffer a stream uses stays referenced until the caller has joined the streams
        pws = workspace(gptq_prepare_workspace_bytes(d), dev)
        U, dm, nd = prepare(H, damp, ws=pws, stream=cons)
        e1 = torch.cuda.Event(enable_timing=True)
        e1.record(cons)
        m_rows = (ctypes.c_int64 * len(Ws))(*[W.shape[0] for W in Ws])
        ws = workspace(max(gptq_quantize_shared_workspace_bytes(len(Ws), m_rows, d, b, block)
                           for b in bits), dev)
        res = {}
        for b in bits:
            res[b] = quantize_shared(Ws, U, b, block, dm, ws=ws, stream=cons)
        e2 = torch.cuda.Event(enable_timing=True)
        e2.record(cons)
        if stage_events is not None:
            stage_events.append(("prepare", e0, e1))
            stage_events.append(("quantize", e1, e2))
        results.append(res)
        n_dead.append(nd)
        keep += [U, dm, ws, pws]   # in use on the consumer streams until the waits below
    if overlap:
        for c in cons_all:
            caller.wait_stream(c)
        caller.wait_stream(prod)
    return results, n_dead


def recon_error(X, W, qpacked, bits, scale, zero, ws=None, stream=None):
    """Per-row ``||(W - W_hat) X^T||^2`` from the packed codes (``[d_out]`` fp32)."""
    torch = _torch()
    n, d = X.shape
    m = W.shape[0]
    if X.stride(1) != 1 or W.stride(1) != 1 or W.shape[1] != d:
        raise ValueError("X [n_tok, d_in] and W [d_out, d_in] must be row-major")
    err = torch.empty(m, dtype=torch.float32, device=W.device)
    if ws is None:
        ws = workspace(gptq_recon_error_workspace_bytes(_dtype_code(X), m, d, n), W.device)
    _check(gptq_recon_error(_ptr(X), _dtype_code(X), n, d, X.stride(0), _ptr(W), _dtype_code(W),
                            m, d if W.stride(0) == d else W.stride(0), _ptr(qpacked), bits,
                            _ptr(scale), _ptr(zero), _ptr(err), _ptr(ws), ws.numel(),
                            _stream(stream)), "gptq_recon_error")
    return err


def quantize_obq(W, U, bits=4, dead_mask=None, ws=None, stream=None):
    """OBQ greedy order per row (d_in <= 128).  Returns
    ``(qpacked, scale, zero, W_hat, order)``."""
    torch = _torch()
    m, d = W.shape
    dev = W.device
    qpacked = torch.empty(m, packed_words(d, bits), dtype=torch.int32, device=dev)
    scale = torch.empty(m, dtype=torch.float32, device=dev)
    zero = torch.empty(m, dtype=torch.int32, device=dev)
    W_hat = torch.empty(m, d, dtype=torch.float32, device=dev)
    order = torch.empty(m, d, dtype=torch.int32, device=dev)
    if ws is None:
        ws = workspace(gptq_quantize_obq_workspace_bytes(m, d), dev)
    _check(gptq_quantize_obq(_ptr(W), _dtype_code(W), m, d, W.stride(0), _ptr(U),
                             _ptr(dead_mask), bits, _ptr(qpacked), _ptr(scale), _ptr(zero),
                             _ptr(W_hat), _ptr(order), _ptr(ws), ws.numel(), _stream(stream)),
           "gptq_quantize_obq")
    return qpacked, scale, zero, W_hat, order
