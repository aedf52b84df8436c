"""gptq_quantize_layer_noalloc: the layer sweep for callers that cannot allocate.

Some callers cannot call cudaMalloc (a host framework that owns the device memory pool,
or code that must not trigger the synchronization an allocation or free can bring).  For
them the library offers a variant of gptq_quantize_layer that takes no workspace and
runs on a fixed scratch array built into the library.  These tests call it through the C
ABI, twice in a row on different layers, and check its outputs against the regular
entry point's on the same inputs; they also check that calls after the first leave the
device's memory untouched, and that the status the call records on the device can be read
back.  The file is named so pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

from oracle import gptq_oracle as O
from post_weight_quantization_03_gb300 import build_lib, gptq
from post_weight_quantization_03_gb300 import synthetic as S

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DT = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib.build()
    gptq.load()
    torch.cuda.init()


def _layer(m, d, wdtype, seed, dead=2):
    # U from the oracle on a synthetic Hessian, W from the seeded generator
    spec = S.ActivationSpec(d_in=d, n_tok=2 * d, dtype="f16", n_dead=dead, n_outlier=1, seed=seed)
    X = S.activations(spec).float().numpy()
    Hd, dmask, _ = O.damp_hessian(O.hessian(X))
    U = torch.from_numpy(O.inverse_cholesky_upper(Hd).astype(np.float32)).to(DEV)
    W = S.weights(m, d, 0.02, wdtype, seed).to(DEV)
    dm = torch.from_numpy(dmask.astype(np.uint8)).to(DEV)
    return W, U, dm


def _outputs(m, d, bits):
    return (torch.empty(m, gptq.packed_words(d, bits), dtype=torch.int32, device=DEV),
            torch.empty(m, dtype=torch.float32, device=DEV),
            torch.empty(m, dtype=torch.int32, device=DEV),
            torch.empty(m, d, dtype=torch.float32, device=DEV))


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(W, U, dm, bits, block, out=None):
    m, d = W.shape
    qp, sc, zr, wh = out if out is not None else _outputs(m, d, bits)
    st = gptq.gptq_quantize_layer_noalloc(_p(W), DT[W.dtype], m, d, W.stride(0), _p(U), _p(dm),
                                          bits, block, _p(qp), _p(sc), _p(zr), _p(wh),
                                          gptq._stream(None))
    assert st == 0, gptq.gptq_status_str(st)
    return qp, sc, zr, wh


def _status():
    return gptq.gptq_noalloc_status(gptq._stream(None))


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    cases = [(256, 384, "bf16", 4, 128, 11), (200, 257, "f32", 3, 128, 12)]
    layers = [_layer(m, d, wdt, seed) for m, d, wdt, _, _, seed in cases]
    # two no-alloc calls in a row on the shared scratch, then the regular entry point
    got = [_noalloc(W, U, dm, c[3], c[4]) for (W, U, dm), c in zip(layers, cases)]
    torch.cuda.synchronize()
    for (W, U, dm), c, g in zip(layers, cases, got):
        ref = gptq.quantize(W, U, c[3], c[4], dm)
        torch.cuda.synchronize()
        for a, b in zip(g, ref):
            assert torch.equal(a, b)     # same kernels, same inputs: identical outputs
    # and once more on the first layer, after the second has left its data in the scratch
    again = _noalloc(*layers[0], cases[0][3], cases[0][4])
    torch.cuda.synchronize()
    for a, b in zip(again, got[0]):
        assert torch.equal(a, b)


def test_noalloc_allocates_nothing_after_the_first_call():
    # eager (B = 1) and blocked sweeps, outputs allocated beforehand: after a warm-up call
    # (which loads the scratch array) neither the device's free memory nor torch's
    # allocator may move across further calls
    W, U, dm = _layer(160, 200, "bf16", 21)
    outs = {blk: _outputs(160, 200, 4) for blk in (1, 128)}
    for blk in (1, 128):
        _noalloc(W, U, dm, 4, blk, outs[blk])
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(2):
        for blk in (1, 128):
            _noalloc(W, U, dm, 4, blk, outs[blk])
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == alloc0
    assert _status() == 0
    for blk in (1, 128):
        ref = gptq.quantize(W, U, 4, blk, dm)
        torch.cuda.synchronize()
        for a, b in zip(outs[blk], ref):
            assert torch.equal(a, b)


def test_noalloc_status_reports_nonfinite_weights():
    W, U, dm = _layer(64, 128, "f32", 31)
    W[5, 17] = float("nan")
    _noalloc(W, U, dm, 4, 128)
    assert _status() == 3          # GPTQ_ERR_NONFINITE
    W[5, 17] = 0.0
    _noalloc(W, U, dm, 4, 128)     # each call clears the status it records
    assert _status() == 0


def test_noalloc_rejects_layers_larger_than_its_scratch():
    m = d = 4096
    need = gptq.gptq_quantize_workspace_bytes(m, d, 4, 128)
    assert need > gptq.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    st = gptq.gptq_quantize_layer_noalloc(fake, 1, m, d, d, fake, None, 4, 128, fake, fake, fake,
                                          None, None)
    assert st == 7  # GPTQ_ERR_WORKSPACE
