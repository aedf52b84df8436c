"""Guard bytes around every buffer the C ABI writes: a stand-in for a memory checker.

Each output and each workspace is the middle of a larger device allocation whose leading
and trailing GUARD bytes hold a fixed pattern.  The calls run through the C ABI on ragged
shapes that take every kernel path (tensor-core and CUDA-core Hessians, the host-streamed
Hessian, the factorization with and without its side streams, the blocked sweep at several
block widths, the eager sweep, the stacked multi-layer sweep, OBQ, the consumer and the
allocation-free sweep); afterwards every guard byte must still hold the pattern, so a store
past a buffer's end fails here instead of corrupting a neighbour.
"""

import ctypes

import pytest
import torch

from post_weight_quantization_03_gb300 import build_lib, gptq
from post_weight_quantization_03_gb300 import synthetic as S

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GUARD = 4096          # bytes each side; a multiple of 256, so the middle keeps that alignment
PAT = 0xA5
DT = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib.build()
    gptq.load()
    torch.cuda.init()


class Guarded:
    """nbytes of device memory between two guard regions holding PAT."""

    def __init__(self, nbytes):
        self.n = int(nbytes)
        self.buf = torch.full((self.n + 2 * GUARD,), PAT, dtype=torch.uint8, device=DEV)
        assert self.buf.data_ptr() % 256 == 0

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr() + GUARD)

    def view(self, dtype, shape):
        return self.buf[GUARD:GUARD + self.n].view(dtype).view(shape)

    def intact(self):
        torch.cuda.synchronize()
        return bool((self.buf[:GUARD] == PAT).all()) and bool((self.buf[GUARD + self.n:] == PAT).all())


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _s():
    return gptq._stream(None)


def _x(d, n, dtype, seed):
    spec = S.ActivationSpec(d_in=d, n_tok=n, dtype=dtype, n_dead=2, n_outlier=1, seed=seed)
    X = S.activations(spec, device=DEV)
    es = X.element_size()
    ld = -(-d * es // 16) * 16 // es      # row pitch a multiple of 16 bytes
    Xp = torch.zeros(n, ld, dtype=X.dtype, device=DEV)
    Xp[:, :d] = X
    return Xp, ld


def _hessian_into(H, X, ld, d, n):
    st = gptq.gptq_hessian_accumulate(_p(X), DT[X.dtype], n, d, ld, H.ptr, 0, _s())
    assert st == 0, gptq.gptq_status_str(st)


@pytest.mark.parametrize("d,n,dtype", [(300, 777, torch.float16), (3998, 512, torch.float16),
                                       (3000, 4100, torch.float16),   # last round cut
                                       (300, 200, torch.float32), (40, 20, torch.float16)])
def test_hessian_stays_in_bounds(d, n, dtype):
    X, ld = _x(d, n, {torch.float16: "f16", torch.float32: "f32"}[dtype], d + n)
    H = Guarded(d * d * 4)
    _hessian_into(H, X, ld, d, n)
    assert H.intact()
    # and accumulating onto it
    st = gptq.gptq_hessian_accumulate(_p(X), DT[X.dtype], n, d, ld, H.ptr, 1, _s())
    assert st == 0 and H.intact()


def test_host_streamed_hessian_stays_in_bounds():
    d, n, chunk = 384, 3000, 1024
    X, ld = _x(d, n, "f16", 5)
    Xh = X.cpu().pin_memory()
    H = Guarded(d * d * 4)
    wsb = gptq.gptq_hessian_host_workspace_bytes(0, d, chunk)
    ws = Guarded(wsb)
    st = gptq.gptq_hessian_accumulate_host(_p(Xh), 0, n, d, ld, H.ptr, 0, chunk, ws.ptr, wsb, _s())
    assert st == 0, gptq.gptq_status_str(st)
    assert H.intact() and ws.intact()


def _prepare(d, seed):
    """A damped factor U of a synthetic Hessian, every buffer guarded."""
    X, ld = _x(d, 2 * d, "f16", seed)
    H = Guarded(d * d * 4)
    _hessian_into(H, X, ld, d, 2 * d)
    U, dm = Guarded(d * d * 4), Guarded(d)
    nd = ctypes.c_int32(-1)                  # n_dead is a host output
    wsb = gptq.gptq_prepare_workspace_bytes(d)
    ws = Guarded(wsb)
    st = gptq.gptq_prepare(H.ptr, d, ctypes.c_float(0.01), U.ptr, dm.ptr,
                           ctypes.c_void_p(ctypes.addressof(nd)), ws.ptr, wsb, _s())
    assert st == 0, gptq.gptq_status_str(st)
    assert nd.value == 2                     # the two dead channels of the synthetic X
    for g in (H, U, dm, ws):
        assert g.intact()
    return U, dm


@pytest.mark.parametrize("d", [300, 512, 1100])   # unaligned: one stream; aligned; a far group
def test_prepare_stays_in_bounds(d):
    U, _ = _prepare(d, 11 + d)
    assert torch.isfinite(U.view(torch.float32, (d, d))).all()


def _outputs(m, d, bits):
    return (Guarded(m * gptq.packed_words(d, bits) * 4), Guarded(m * 4), Guarded(m * 4),
            Guarded(m * d * 4))


@pytest.mark.parametrize("m,d,bits,block", [(131, 300, 3, 128), (64, 257, 4, 32),
                                            (70, 150, 2, 7), (33, 65, 8, 1), (200, 600, 4, 128)])
def test_quantize_stays_in_bounds(m, d, bits, block):
    U, dm = _prepare(d, 3 * d + m)
    W = S.weights(m, d, 0.02, "bf16", m + d).to(DEV)
    qp, sc, zr, wh = _outputs(m, d, bits)
    wsb = gptq.gptq_quantize_workspace_bytes(m, d, bits, block)
    ws = Guarded(wsb)
    st = gptq.gptq_quantize_layer(_p(W), 1, m, d, W.stride(0), U.ptr, dm.ptr, bits, block,
                                  qp.ptr, sc.ptr, zr.ptr, wh.ptr, ws.ptr, wsb, _s())
    assert st == 0, gptq.gptq_status_str(st)
    assert gptq.gptq_workspace_status(ws.ptr, _s()) == 0
    for g in (qp, sc, zr, wh, ws, U, dm):
        assert g.intact()


def test_shared_sweep_stays_in_bounds():
    d, bits, block, ms = 300, 4, 128, (50, 77)
    U, dm = _prepare(d, 41)
    Ws = [S.weights(m, d, 0.02, "f16", 50 + m).to(DEV) for m in ms]
    outs = [_outputs(m, d, bits) for m in ms]
    n = len(ms)
    rows = (ctypes.c_int64 * n)(*ms)
    wsb = gptq.gptq_quantize_shared_workspace_bytes(n, rows, d, bits, block)
    ws = Guarded(wsb)
    P = ctypes.c_void_p
    st = gptq.gptq_quantize_layers_shared(
        n, (P * n)(*[W.data_ptr() for W in Ws]), (ctypes.c_int * n)(*[0] * n), rows,
        (ctypes.c_int64 * n)(*[W.stride(0) for W in Ws]), d, U.ptr, dm.ptr, bits, block,
        (P * n)(*[o[0].ptr.value for o in outs]), (P * n)(*[o[1].ptr.value for o in outs]),
        (P * n)(*[o[2].ptr.value for o in outs]), (P * n)(*[o[3].ptr.value for o in outs]),
        ws.ptr, wsb, _s())
    assert st == 0, gptq.gptq_status_str(st)
    assert ws.intact()
    for o in outs:
        for g in o:
            assert g.intact()


def test_obq_stays_in_bounds():
    m, d, bits = 50, 100, 4
    U, dm = _prepare(d, 61)
    W = S.weights(m, d, 0.02, "bf16", 62).to(DEV)
    qp, sc, zr, wh = _outputs(m, d, bits)
    order = Guarded(m * d * 4)
    wsb = gptq.gptq_quantize_obq_workspace_bytes(m, d)
    ws = Guarded(wsb)
    st = gptq.gptq_quantize_obq(_p(W), 1, m, d, W.stride(0), U.ptr, dm.ptr, bits, qp.ptr,
                                sc.ptr, zr.ptr, wh.ptr, order.ptr, ws.ptr, wsb, _s())
    assert st == 0, gptq.gptq_status_str(st)
    for g in (qp, sc, zr, wh, order, ws):
        assert g.intact()


@pytest.mark.parametrize("xdtype", ["f16", "f32"])
def test_recon_error_stays_in_bounds(xdtype):
    m, d, n, bits = 70, 264, 700, 4
    U, dm = _prepare(d, 71)
    W = S.weights(m, d, 0.02, "bf16", 72).to(DEV)
    qp, sc, zr, wh = _outputs(m, d, bits)
    wsq = gptq.gptq_quantize_workspace_bytes(m, d, bits, 128)
    wq = Guarded(wsq)
    assert gptq.gptq_quantize_layer(_p(W), 1, m, d, W.stride(0), U.ptr, dm.ptr, bits, 128,
                                    qp.ptr, sc.ptr, zr.ptr, wh.ptr, wq.ptr, wsq, _s()) == 0
    X, ld = _x(d, n, xdtype, 73)
    err = Guarded(m * 4)
    wsb = gptq.gptq_recon_error_workspace_bytes(DT[X.dtype], m, d, n)
    ws = Guarded(wsb)
    st = gptq.gptq_recon_error(_p(X), DT[X.dtype], n, d, ld, _p(W), 1, m, W.stride(0), qp.ptr,
                               bits, sc.ptr, zr.ptr, err.ptr, ws.ptr, wsb, _s())
    assert st == 0, gptq.gptq_status_str(st)
    for g in (err, ws, qp, sc, zr):
        assert g.intact()
    assert torch.isfinite(err.view(torch.float32, (m,))).all()


def test_noalloc_sweep_stays_in_bounds():
    m, d, bits = 96, 200, 3
    U, dm = _prepare(d, 81)
    W = S.weights(m, d, 0.02, "f16", 82).to(DEV)
    qp, sc, zr, wh = _outputs(m, d, bits)
    st = gptq.gptq_quantize_layer_noalloc(_p(W), 0, m, d, W.stride(0), U.ptr, dm.ptr, bits, 128,
                                          qp.ptr, sc.ptr, zr.ptr, wh.ptr, _s())
    assert st == 0, gptq.gptq_status_str(st)
    assert gptq.gptq_noalloc_status(_s()) == 0
    for g in (qp, sc, zr, wh):
        assert g.intact()
    # the guarded outputs hold what the workspace entry point computes
    ref = gptq.quantize(W, U.view(torch.float32, (d, d)), bits, 128, dm.view(torch.uint8, (d,)))
    torch.cuda.synchronize()
    assert torch.equal(qp.view(torch.int32, ref[0].shape), ref[0])
    assert torch.equal(wh.view(torch.float32, (m, d)), ref[3])
