"""The factorization and the sweep replay captured graphs of their launches (one per buffer
set, a few kept): these tests check that replays compute what the first call computed, on
any stream, when more buffer sets are used than are kept, and when the caller captures the
sweep into a graph of their own.

The sweep is deterministic (bit-identical across calls and schedules); the factorization
adds into shared blocks from two streams, so its repeats are compared with the oracle and
with each other to fp32 rounding.
"""

import numpy as np
import pytest
import torch

from oracle import gptq_oracle as O
from post_weight_quantization_03_gb300 import build_lib, gptq
from post_weight_quantization_03_gb300 import synthetic as S
from tests import parity as PT

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib.build()
    gptq.load()
    torch.cuda.init()


def _problem(d, seed, n=None):
    spec = S.ActivationSpec(d_in=d, n_tok=n or 3 * d, dtype="f16", n_dead=2, n_outlier=1,
                            seed=seed)
    X = S.activations(spec)
    H64 = O.hessian(X.float().numpy())
    Ur = O.inverse_cholesky_upper(O.damp_hessian(H64)[0])
    return X, H64.astype(np.float32), Ur


def test_factorization_replays_match_the_oracle_on_any_stream():
    d = 512
    _, H32, Ur = _problem(d, 3)
    Hsrc = torch.from_numpy(H32).to(DEV)
    H = torch.empty_like(Hsrc)
    U = torch.empty_like(Hsrc)
    dm = torch.empty(d, dtype=torch.uint8, device=DEV)
    ws = gptq.workspace(gptq.gptq_prepare_workspace_bytes(d), DEV)
    side = torch.cuda.Stream(DEV)
    outs = []
    for rep in range(4):                     # first call captures, the others replay
        st = side if rep % 2 else None       # the legacy default stream and another one
        with torch.cuda.stream(st) if st is not None else torch.cuda.stream(
                torch.cuda.current_stream()):
            H.copy_(Hsrc)
            gptq.prepare(H, 0.01, U=U, dead_mask=dm, ws=ws)
        torch.cuda.synchronize()
        got = U.cpu().numpy()
        assert PT.u_rowwise_err(got, Ur) <= PT.TOL_U
        outs.append(got)
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) <= 1e-5 * np.max(np.abs(outs[0]))


def test_more_buffer_sets_than_kept_graphs():
    # ten distinct (H, U, workspace) sets, used twice each in an interleaved order
    d = 256
    cases = [_problem(d, 10 + i) for i in range(10)]
    bufs = [(torch.empty(d, d, device=DEV), torch.empty(d, d, device=DEV),
             gptq.workspace(gptq.gptq_prepare_workspace_bytes(d), DEV)) for _ in cases]
    for rnd in range(2):
        for (_, H32, Ur), (H, U, ws) in zip(cases, bufs):
            H.copy_(torch.from_numpy(H32).to(DEV))
            gptq.prepare(H, 0.01, U=U, ws=ws)
            torch.cuda.synchronize()
            assert PT.u_rowwise_err(U.cpu().numpy(), Ur) <= PT.TOL_U


def test_sweep_replays_are_bit_identical_and_match_separate_buffers():
    d, m, bits = 512, 300, 4
    _, H32, Ur = _problem(d, 21)
    U = torch.from_numpy(Ur.astype(np.float32)).to(DEV)
    W = S.weights(m, d, 0.02, "bf16", 22).to(DEV)
    ws = gptq.workspace(gptq.gptq_quantize_workspace_bytes(m, d, bits, 128), DEV)
    out = (torch.empty(m, gptq.packed_words(d, bits), dtype=torch.int32, device=DEV),
           torch.empty(m, dtype=torch.float32, device=DEV),
           torch.empty(m, dtype=torch.int32, device=DEV),
           torch.empty(m, d, dtype=torch.float32, device=DEV))
    ref = [t.clone() for t in gptq.quantize(W, U, bits, 128)]    # fresh buffers
    side = torch.cuda.Stream(DEV)
    for rep in range(3):
        with torch.cuda.stream(side if rep == 1 else torch.cuda.current_stream()):
            for t in out:
                t.zero_()
            gptq.quantize(W, U, bits, 128, ws=ws, out=out)
        torch.cuda.synchronize()
        for a, b in zip(out, ref):
            assert torch.equal(a, b)


def test_sweep_inside_the_callers_graph_capture():
    d, m, bits = 384, 200, 3
    _, H32, Ur = _problem(d, 31)
    U = torch.from_numpy(Ur.astype(np.float32)).to(DEV)
    W = S.weights(m, d, 0.02, "bf16", 32).to(DEV)
    ws = gptq.workspace(gptq.gptq_quantize_workspace_bytes(m, d, bits, 128), DEV)
    out = (torch.empty(m, gptq.packed_words(d, bits), dtype=torch.int32, device=DEV),
           torch.empty(m, dtype=torch.float32, device=DEV),
           torch.empty(m, dtype=torch.int32, device=DEV),
           torch.empty(m, d, dtype=torch.float32, device=DEV))
    ref = [t.clone() for t in gptq.quantize(W, U, bits, 128)]
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(DEV)
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        gptq.quantize(W, U, bits, 128, ws=ws, out=out)        # warm-up outside the capture
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=cap):
        gptq.quantize(W, U, bits, 128, ws=ws, out=out)
    for t in out:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(out, ref):
        assert torch.equal(a, b)
